"""Packed variable-length attention (head_dim 64) for one GB300 (sm_103a).

Thin Python binding over the C ABI of ``libkime_attn.so`` (declared in
``include/kime_attn.h``).  Every function here only marshals arguments: it
reads shapes, data pointers and the current CUDA stream from torch tensors,
allocates outputs / scratch with torch when the caller passes none, and calls
the C entry point of the same name.  All arithmetic runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If the shared library has not
been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "KimeError", "load_library", "kime_attn_varlen", "kime_kv_append", "kime_attn_decode",
    "kime_attn_workspace_bytes", "kime_rope_tables", "kime_attn_debug_tiles", "kime_attn_varlen_noalloc",
    "kime_decode_step", "kime_kv_append_varlen", "kime_attn_chunk", "kime_chunk_step",
    "kime_attn_debug_tiles_chunk", "KIME_F32", "KIME_BF16", "KIME_F32_3XTF32", "EXPORTED_SYMBOLS",
    "NOALLOC_SCRATCH_BYTES",
    "kime_qkv_proj", "kime_attn_varlen_proj",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkime_attn.so")

KIME_F32, KIME_BF16, KIME_F32_F16OUT, KIME_F32_BF16OUT, KIME_F32_3XTF32 = 0, 1, 2, 3, 4
DEV_BAD_CU, DEV_SEQ_TOO_LONG, DEV_BAD_POS, DEV_TIMEOUT, DEV_RANGE = 1, 2, 4, 8, 16

EXPORTED_SYMBOLS = (
    "kime_attn_varlen", "kime_kv_append", "kime_attn_decode", "kime_attn_workspace_bytes",
    "kime_rope_tables", "kime_attn_debug_tiles", "kime_attn_last_cuda_error", "kime_attn_status_string",
    "kime_attn_varlen_noalloc", "kime_decode_step", "kime_kv_append_varlen", "kime_attn_chunk",
    "kime_chunk_step", "kime_attn_debug_tiles_chunk", "kime_qkv_proj", "kime_attn_varlen_proj",
)
NOALLOC_SCRATCH_BYTES = 1 << 20

_lib = None


class KimeError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str, cuda_error: int = 0):
        super().__init__(f"{fn} failed: {msg} (status {status}, cuda error {cuda_error})")
        self.status = status
        self.cuda_error = cuda_error


def load_library(path: str = LIB_PATH):
    """Load libkime_attn.so (built by ``build.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkime_attn.so not found at {path}: build it with "
                           "packed_varlen_attention_kime_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F, D, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
    lib.kime_attn_varlen.argtypes = [P, I, P, I, I, I, I, I, I, I, I, F, P, P, I, P, P, S, P, P]
    lib.kime_attn_varlen.restype = I
    lib.kime_kv_append.argtypes = [P, P, I, I, I, I, I, P, P, I, P, P, P, P]
    lib.kime_kv_append.restype = I
    lib.kime_attn_decode.argtypes = [P, P, I, I, I, I, I, F, P, P, I, P, P, P, P, S, P, P]
    lib.kime_attn_decode.restype = I
    lib.kime_attn_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.kime_attn_workspace_bytes.restype = S
    lib.kime_rope_tables.argtypes = [D, I, P, P]
    lib.kime_rope_tables.restype = I
    lib.kime_attn_debug_tiles.argtypes = [P, I, I, I, I, I, P, S, P, I, P, P, P]
    lib.kime_attn_debug_tiles.restype = I
    lib.kime_decode_step.argtypes = [P, P, I, I, I, I, I, F, P, P, I, P, P, P, P, S, P, P]
    lib.kime_decode_step.restype = I
    lib.kime_attn_varlen_noalloc.argtypes = [P, I, P, I, I, I, I, I, I, I, I, F, P, P, I, P, P, P]
    lib.kime_attn_varlen_noalloc.restype = I
    lib.kime_kv_append_varlen.argtypes = [P, P, P, I, I, I, I, I, I, P, P, I, P, P, P, P]
    lib.kime_kv_append_varlen.restype = I
    lib.kime_attn_chunk.argtypes = [P, P, P, I, I, I, I, I, I, I, F, P, P, I, P, P, P, P, S, P, P]
    lib.kime_attn_chunk.restype = I
    lib.kime_chunk_step.argtypes = [P, P, P, I, I, I, I, I, I, I, F, P, P, I, P, P, P, P, S, P, P]
    lib.kime_chunk_step.restype = I
    lib.kime_attn_debug_tiles_chunk.argtypes = [P, P, I, I, I, I, I, P, S, P, I, P, P, P]
    lib.kime_attn_debug_tiles_chunk.restype = I
    lib.kime_qkv_proj.argtypes = [P, P, I, I, I, I, I, P, P, P]
    lib.kime_qkv_proj.restype = I
    lib.kime_attn_varlen_proj.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, I, P, P, S, P, P]
    lib.kime_attn_varlen_proj.restype = I
    lib.kime_attn_last_cuda_error.argtypes = []
    lib.kime_attn_last_cuda_error.restype = I
    lib.kime_attn_status_string.argtypes = [I]
    lib.kime_attn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != 0:
        lib = load_library()
        raise KimeError(fn, rc, lib.kime_attn_status_string(rc).decode(), lib.kime_attn_last_cuda_error())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(qkv: torch.Tensor, out_dtype, precision=None) -> int:
    """kime_dtype of (qkv, out): same type, or FP32 qkv with a 16-bit output;
    precision="3xtf32" selects FP32 on the tensor cores (FP32 qkv and out)."""
    if precision == "3xtf32":
        if qkv.dtype == torch.float32 and out_dtype == torch.float32:
            return KIME_F32_3XTF32
        raise TypeError(f"3xTF32 needs float32 qkv and out, got {qkv.dtype} -> {out_dtype}")
    if precision is not None:
        raise ValueError(f"unknown precision {precision!r}")
    if qkv.dtype == torch.bfloat16 and out_dtype == torch.bfloat16:
        return KIME_BF16
    if qkv.dtype == torch.float32:
        codes = {torch.float32: KIME_F32, torch.float16: KIME_F32_F16OUT, torch.bfloat16: KIME_F32_BF16OUT}
        if out_dtype in codes:
            return codes[out_dtype]
    raise TypeError(f"unsupported qkv/out dtypes {qkv.dtype} -> {out_dtype}")


def kime_attn_workspace_bytes(op: int, n_seqs: int, total_tokens: int = 0, heads: int = 1,
                              kv_heads: int = 1, cap: int = 1) -> int:
    return int(load_library().kime_attn_workspace_bytes(op, n_seqs, total_tokens, heads, kv_heads, cap))


def kime_rope_tables(theta: float, length: int):
    """cos, sin float32 CPU tensors [length, 32] (kime-cuda ``rope_tables`` recipe)."""
    lib = load_library()
    c = torch.empty((length, 32), dtype=torch.float32)
    s = torch.empty((length, 32), dtype=torch.float32)
    _check("kime_rope_tables", lib.kime_rope_tables(float(theta), int(length), _p(c), _p(s)))
    return c, s


def kime_attn_varlen(qkv, cu_seqlens, max_seqlen, heads, kv_heads, window, causal, scale,
                     rope_cos, rope_sin, out=None, workspace=None, dev_status=None, stream=None, out_dtype=None,
                     precision=None):
    """Attention over the packed batch; returns ``out`` [T, heads*64].  Its
    dtype is qkv's, or (FP32 qkv) float16 / bfloat16 when ``out`` or
    ``out_dtype`` says so.  ``precision="3xtf32"`` (FP32 qkv and out) runs the
    FP32 attention on the tensor cores as three TF32 products."""
    lib = load_library()
    T = qkv.shape[0]
    n_seqs = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, heads * 64), dtype=out_dtype or qkv.dtype, device=qkv.device)
    code = _dtype_code(qkv, out.dtype, precision)
    if workspace is None:
        # BF16 qkv: room for the prepared rows, which the faster kernel reads
        op = 3 if qkv.dtype == torch.bfloat16 else (4 if code == KIME_F32_3XTF32 else 0)
        need = kime_attn_workspace_bytes(op, n_seqs, T, heads, kv_heads)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qkv.device)
    rc = lib.kime_attn_varlen(_p(qkv), code, _p(cu_seqlens), n_seqs, T, int(max_seqlen), heads,
                              kv_heads, 64, int(window), int(bool(causal)), float(scale), _p(rope_cos),
                              _p(rope_sin), rope_cos.shape[0], _p(out), _p(workspace),
                              workspace.numel() * workspace.element_size(), _p(dev_status),
                              _stream(stream, qkv.device))
    _check("kime_attn_varlen", rc)
    return out


def kime_qkv_proj(x, w, heads, kv_heads, out=None, dev_status=None, stream=None):
    """qkv = x w^T (bf16 x [T, hidden], bf16 w [64*(heads+2*kv_heads), hidden]);
    returns bf16 qkv [T, 64*(heads+2*kv_heads)]."""
    lib = load_library()
    T, hidden = x.shape
    if out is None:
        out = torch.empty((T, w.shape[0]), dtype=torch.bfloat16, device=x.device)
    rc = lib.kime_qkv_proj(_p(x), _p(w), T, hidden, heads, kv_heads, 64, _p(out), _p(dev_status),
                           _stream(stream, x.device))
    _check("kime_qkv_proj", rc)
    return out


def kime_attn_varlen_proj(x, w, cu_seqlens, max_seqlen, heads, kv_heads, window, causal, scale, rope_cos,
                          rope_sin, out=None, workspace=None, dev_status=None, stream=None):
    """Attention over the packed batch whose qkv rows are x w^T, the projection
    fused into the attention's producer; returns bf16 out [T, heads*64]."""
    lib = load_library()
    T, hidden = x.shape
    n_seqs = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, heads * 64), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        need = kime_attn_workspace_bytes(3, n_seqs, T, heads, kv_heads)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    rc = lib.kime_attn_varlen_proj(_p(x), _p(w), _p(cu_seqlens), n_seqs, T, hidden, int(max_seqlen), heads,
                                   kv_heads, 64, int(window), int(bool(causal)), float(scale), _p(rope_cos),
                                   _p(rope_sin), rope_cos.shape[0], _p(out), _p(workspace),
                                   workspace.numel() * workspace.element_size(), _p(dev_status),
                                   _stream(stream, x.device))
    _check("kime_attn_varlen_proj", rc)
    return out


def kime_attn_varlen_noalloc(qkv, cu_seqlens, max_seqlen, heads, kv_heads, window, causal, scale,
                             rope_cos, rope_sin, out=None, dev_status=None, stream=None):
    """kime_attn_varlen without a caller-provided scratch buffer: for callers
    that cannot allocate device memory at call time.  The C entry point uses a
    fixed scratch array built into the library (NOALLOC_SCRATCH_BYTES), shared
    by all calls -- calls that overlap on the GPU race.  Only `out`, if not
    given, is allocated here by torch."""
    lib = load_library()
    T = qkv.shape[0]
    n_seqs = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, heads * 64), dtype=qkv.dtype, device=qkv.device)
    rc = lib.kime_attn_varlen_noalloc(_p(qkv), _dtype_code(qkv, out.dtype), _p(cu_seqlens), n_seqs, T, int(max_seqlen),
                                      heads, kv_heads, 64, int(window), int(bool(causal)), float(scale),
                                      _p(rope_cos), _p(rope_sin), rope_cos.shape[0], _p(out), _p(dev_status),
                                      _stream(stream, qkv.device))
    _check("kime_attn_varlen_noalloc", rc)
    return out


def kime_kv_append(qkv_new, pos, heads, kv_heads, k_cache, v_cache, rope_cos, rope_sin,
                   dev_status=None, stream=None):
    """Writes the new token's RoPE'd k and its v at row pos[s] of the caches."""
    lib = load_library()
    cap = k_cache.shape[2]
    rc = lib.kime_kv_append(_p(qkv_new), _p(pos), pos.numel(), heads, kv_heads, 64, cap, _p(rope_cos),
                            _p(rope_sin), rope_cos.shape[0], _p(k_cache), _p(v_cache), _p(dev_status),
                            _stream(stream, qkv_new.device))
    _check("kime_kv_append", rc)


def kime_attn_decode(qkv_new, pos, heads, kv_heads, k_cache, v_cache, scale, rope_cos, rope_sin,
                     out=None, workspace=None, dev_status=None, stream=None):
    """Single-token attention of each sequence's new row over cache rows 0..=pos[s]."""
    lib = load_library()
    n = pos.numel()
    cap = k_cache.shape[2]
    if out is None:
        out = torch.empty((n, heads * 64), dtype=torch.bfloat16, device=qkv_new.device)
    need = kime_attn_workspace_bytes(1, n, 0, heads, kv_heads, cap)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qkv_new.device)
    rc = lib.kime_attn_decode(_p(qkv_new), _p(pos), n, heads, kv_heads, 64, cap, float(scale),
                              _p(rope_cos), _p(rope_sin), rope_cos.shape[0], _p(k_cache), _p(v_cache),
                              _p(out), _p(workspace), workspace.numel() * workspace.element_size(),
                              _p(dev_status), _stream(stream, qkv_new.device))
    _check("kime_attn_decode", rc)
    return out


def kime_decode_step(qkv_new, pos, heads, kv_heads, k_cache, v_cache, scale, rope_cos, rope_sin,
                     out=None, workspace=None, dev_status=None, stream=None):
    """KV append and single-token decode in one launch; returns ``out``."""
    lib = load_library()
    n = pos.numel()
    cap = k_cache.shape[2]
    if out is None:
        out = torch.empty((n, heads * 64), dtype=torch.bfloat16, device=qkv_new.device)
    need = kime_attn_workspace_bytes(1, n, 0, heads, kv_heads, cap)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qkv_new.device)
    rc = lib.kime_decode_step(_p(qkv_new), _p(pos), n, heads, kv_heads, 64, cap, float(scale),
                              _p(rope_cos), _p(rope_sin), rope_cos.shape[0], _p(k_cache), _p(v_cache),
                              _p(out), _p(workspace), workspace.numel() * workspace.element_size(),
                              _p(dev_status), _stream(stream, qkv_new.device))
    _check("kime_decode_step", rc)
    return out


def kime_attn_debug_tiles(cu_seqlens, total_tokens, max_seqlen, window, causal, dev_status=None,
                          stream=None):
    """The scheduler's work list: int32 [n_pairs, 8] rows of
    (s, qt, kt_begin, kt_end, full_begin, full_end, row0, L), on the device."""
    lib = load_library()
    n_seqs = cu_seqlens.numel() - 1
    dev = cu_seqlens.device
    max_pairs = total_tokens // 128 + n_seqs + 1
    need = kime_attn_workspace_bytes(0, n_seqs, total_tokens)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    tiles = torch.zeros((max_pairs, 8), dtype=torch.int32, device=dev)
    count = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.kime_attn_debug_tiles(_p(cu_seqlens), n_seqs, int(total_tokens), int(max_seqlen), int(window),
                                   int(bool(causal)), _p(ws), need, _p(tiles), max_pairs, _p(count),
                                   _p(dev_status), _stream(stream, dev))
    _check("kime_attn_debug_tiles", rc)
    n = int(count.item())
    return tiles[:n]


def kime_kv_append_varlen(qkv, cu_seqlens, pos, heads, kv_heads, k_cache, v_cache, rope_cos, rope_sin,
                          dev_status=None, stream=None):
    """Writes row i of each sequence's block (RoPE'd k, v) at cache row pos[s] + i."""
    lib = load_library()
    cap = k_cache.shape[2]
    rc = lib.kime_kv_append_varlen(_p(qkv), _p(cu_seqlens), _p(pos), pos.numel(), qkv.shape[0], heads, kv_heads,
                                   64, cap, _p(rope_cos), _p(rope_sin), rope_cos.shape[0], _p(k_cache),
                                   _p(v_cache), _p(dev_status), _stream(stream, qkv.device))
    _check("kime_kv_append_varlen", rc)


def _chunk(fn, qkv, cu_seqlens, pos, max_seqlen, heads, kv_heads, k_cache, v_cache, scale, rope_cos, rope_sin,
           out, workspace, dev_status, stream):
    lib = load_library()
    T = qkv.shape[0]
    n = pos.numel()
    cap = k_cache.shape[2]
    if out is None:
        out = torch.empty((T, heads * 64), dtype=torch.bfloat16, device=qkv.device)
    # room for the prepared rows (op 5): the faster path; any workspace of at
    # least kime_attn_workspace_bytes(2, ...) bytes is accepted
    need = kime_attn_workspace_bytes(5, n, T, heads, kv_heads, cap)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qkv.device)
    rc = getattr(lib, fn)(_p(qkv), _p(cu_seqlens), _p(pos), n, T, int(max_seqlen), heads, kv_heads, 64, cap,
                          float(scale), _p(rope_cos), _p(rope_sin), rope_cos.shape[0], _p(k_cache), _p(v_cache),
                          _p(out), _p(workspace), workspace.numel() * workspace.element_size(), _p(dev_status),
                          _stream(stream, qkv.device))
    _check(fn, rc)
    return out


def kime_attn_chunk(qkv, cu_seqlens, pos, max_seqlen, heads, kv_heads, k_cache, v_cache, scale, rope_cos,
                    rope_sin, out=None, workspace=None, dev_status=None, stream=None):
    """Chunked-prefill attention: row i of sequence s attends cache rows
    0..pos[s]+i (the caches already hold the chunk); returns ``out``."""
    return _chunk("kime_attn_chunk", qkv, cu_seqlens, pos, max_seqlen, heads, kv_heads, k_cache, v_cache, scale,
                  rope_cos, rope_sin, out, workspace, dev_status, stream)


def kime_chunk_step(qkv, cu_seqlens, pos, max_seqlen, heads, kv_heads, k_cache, v_cache, scale, rope_cos,
                    rope_sin, out=None, workspace=None, dev_status=None, stream=None):
    """kime_kv_append_varlen then kime_attn_chunk; returns ``out``."""
    return _chunk("kime_chunk_step", qkv, cu_seqlens, pos, max_seqlen, heads, kv_heads, k_cache, v_cache, scale,
                  rope_cos, rope_sin, out, workspace, dev_status, stream)


def kime_attn_debug_tiles_chunk(cu_seqlens, pos, total_tokens, max_seqlen, cap, rope_len, dev_status=None,
                                stream=None):
    """The scheduler's work list for chunks at offsets pos (causal): int32
    [n_pairs, 8] rows of (s, qt, kt_begin, kt_end, full_begin, full_end, row0, L)."""
    lib = load_library()
    n_seqs = cu_seqlens.numel() - 1
    dev = cu_seqlens.device
    max_pairs = total_tokens // 128 + n_seqs + 1
    need = kime_attn_workspace_bytes(2, n_seqs, total_tokens)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    tiles = torch.zeros((max_pairs, 8), dtype=torch.int32, device=dev)
    count = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.kime_attn_debug_tiles_chunk(_p(cu_seqlens), _p(pos), n_seqs, int(total_tokens), int(max_seqlen),
                                         int(cap), int(rope_len), _p(ws), need, _p(tiles), max_pairs, _p(count),
                                         _p(dev_status), _stream(stream, dev))
    _check("kime_attn_debug_tiles_chunk", rc)
    n = int(count.item())
    return tiles[:n]
