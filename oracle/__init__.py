"""FP64 CPU oracle for packed variable-length attention with RoPE.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of ``bench.py`` may import this package; the
product path (``packed_varlen_attention_kime_gb300``) never does.  The oracle
shares no code with the CUDA library; it is a thin ctypes wrapper over
``kime_oracle.c`` (plain C, double precision, threaded over independent
queries) plus the brute-force tile classifier in ``tiles.py``.

Inputs are numpy arrays.  bfloat16 data is passed as its uint16 bit patterns
(widened exactly inside the oracle).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kime_oracle.c")
_LIB = os.path.join(_HERE, "libkime_oracle.so")
_lib = None

DT_F64, DT_F32, DT_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add: the KV append's
    float32 rotation must round after every operation)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, I, D, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.kime_oracle_rope_tables_f32.argtypes = [D, I, P, P]
        lib.kime_oracle_rope_tables_f64.argtypes = [D, I, P, P]
        lib.kime_oracle_rope.argtypes = [P, P, P, P]
        lib.kime_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.kime_oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.kime_oracle_attn_varlen.argtypes = [P, I, P, I, I, I, I, I, D, P, P, I, P, P, L, P, I, I]
        lib.kime_oracle_attn_varlen.restype = I
        lib.kime_oracle_attn_probs.argtypes = [P, I, P, I, I, I, I, I, D, P, P, I, I, I, P, I]
        lib.kime_oracle_attn_probs.restype = I
        lib.kime_oracle_kv_append.argtypes = [P, P, I, I, I, I, P, P, I, P, P]
        lib.kime_oracle_kv_append.restype = I
        lib.kime_oracle_attn_decode.argtypes = [P, P, I, I, I, I, D, P, P, I, P, P, P, L, P, I]
        lib.kime_oracle_attn_decode.restype = I
        lib.kime_oracle_kv_append_varlen.argtypes = [P, P, P, I, I, I, I, P, P, I, P, P]
        lib.kime_oracle_kv_append_varlen.restype = I
        lib.kime_oracle_attn_chunk.argtypes = [P, P, P, I, I, I, I, D, P, P, I, P, P, P, P, L, P, I]
        lib.kime_oracle_attn_chunk.restype = I
        lib.kime_oracle_qkv_proj.argtypes = [P, P, I, I, I, P, I]
        lib.kime_oracle_qkv_proj.restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _data(qkv):
    """(contiguous array, dtype code).  uint16 arrays are bfloat16 bits."""
    qkv = np.ascontiguousarray(qkv)
    if qkv.dtype == np.float64:
        return qkv, DT_F64
    if qkv.dtype == np.float32:
        return qkv, DT_F32
    if qkv.dtype == np.uint16:
        return qkv, DT_BF16
    raise TypeError(f"unsupported qkv dtype {qkv.dtype}")


def rope_tables_f32(theta: float, length: int):
    """cos, sin float32 [length, 32] by the kime-cuda ``rope_tables`` recipe."""
    lib = _load()
    c = np.zeros((length, 32), np.float32)
    s = np.zeros((length, 32), np.float32)
    lib.kime_oracle_rope_tables_f32(float(theta), int(length), _ptr(c), _ptr(s))
    return c, s


def rope_tables_f64(theta: float, length: int):
    """cos, sin float64 [length, 32] with exact double angles."""
    lib = _load()
    c = np.zeros((length, 32), np.float64)
    s = np.zeros((length, 32), np.float64)
    lib.kime_oracle_rope_tables_f64(float(theta), int(length), _ptr(c), _ptr(s))
    return c, s


def rope(x, cos_row, sin_row):
    """Rotate-half RoPE of one 64-vector with one table row (all float64)."""
    lib = _load()
    x = np.ascontiguousarray(x, np.float64)
    c = np.ascontiguousarray(cos_row, np.float64)
    s = np.ascontiguousarray(sin_row, np.float64)
    y = np.zeros(64, np.float64)
    lib.kime_oracle_rope(_ptr(x), _ptr(c), _ptr(s), _ptr(y))
    return y


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    lib = _load()
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib.kime_oracle_f32_to_bf16(float(v)) for v in x], np.uint16)


def attn_varlen(qkv, cu, heads, kv_heads, window, causal, scale, cos, sin, rows=None,
                row_heads=None, mode=0, nthreads=None):
    """Attention outputs in float64.

    rows=None: every row and head, returned as [T, heads*64].
    rows / row_heads given: outputs of those (token row, head) pairs, [n, 64].
    mode 0 skips masked keys; mode 1 materialises -inf and takes softmax of the
    whole row.  cos/sin are float64 (widen float32 tables exactly).
    """
    lib = _load()
    qkv, dt = _data(qkv)
    cu = np.ascontiguousarray(cu, np.int32)
    n_seqs = len(cu) - 1
    cos = np.ascontiguousarray(cos, np.float64)
    sin = np.ascontiguousarray(sin, np.float64)
    if rows is None:
        T = int(cu[-1]) if n_seqs > 0 else 0
        out = np.zeros((T, heads * 64), np.float64)
        n_items = T * heads
        rp = hp = None
    else:
        rows = np.ascontiguousarray(rows, np.int32)
        row_heads = np.ascontiguousarray(row_heads, np.int32)
        n_items = len(rows)
        out = np.zeros((n_items, 64), np.float64)
        rp, hp = rows, row_heads
    rc = lib.kime_oracle_attn_varlen(_ptr(qkv), dt, _ptr(cu), n_seqs, heads, kv_heads, window,
                                     int(bool(causal)), float(scale), _ptr(cos), _ptr(sin),
                                     cos.shape[0], _ptr(rp), _ptr(hp), n_items, _ptr(out), mode,
                                     _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def attn_probs(qkv, cu, heads, kv_heads, window, causal, scale, cos, sin, row, head, mode=0):
    """The probability row of query (row, head): length L of its sequence."""
    lib = _load()
    qkv, dt = _data(qkv)
    cu = np.ascontiguousarray(cu, np.int32)
    n_seqs = len(cu) - 1
    s = int(np.searchsorted(cu, row, side="right") - 1)
    s = min(s, n_seqs - 1)
    L = int(cu[s + 1] - cu[s])
    cos = np.ascontiguousarray(cos, np.float64)
    sin = np.ascontiguousarray(sin, np.float64)
    probs = np.zeros(max(L, 1), np.float64)
    rc = lib.kime_oracle_attn_probs(_ptr(qkv), dt, _ptr(cu), n_seqs, heads, kv_heads, window,
                                    int(bool(causal)), float(scale), _ptr(cos), _ptr(sin),
                                    cos.shape[0], int(row), int(head), _ptr(probs), mode)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return probs[:L]


def kv_append(qkv_new_bits, pos, heads, kv_heads, cap, cos32, sin32, k_cache_bits, v_cache_bits):
    """In-place append into uint16 (bfloat16 bits) caches [n, kv_heads, cap, 64].
    Returns the number of sequences skipped for an out-of-range pos."""
    lib = _load()
    q = np.ascontiguousarray(qkv_new_bits, np.uint16)
    pos = np.ascontiguousarray(pos, np.int32)
    c = np.ascontiguousarray(cos32, np.float32)
    s = np.ascontiguousarray(sin32, np.float32)
    assert k_cache_bits.dtype == np.uint16 and k_cache_bits.flags.c_contiguous
    assert v_cache_bits.dtype == np.uint16 and v_cache_bits.flags.c_contiguous
    return lib.kime_oracle_kv_append(_ptr(q), _ptr(pos), len(pos), heads, kv_heads, cap, _ptr(c),
                                     _ptr(s), c.shape[0], _ptr(k_cache_bits), _ptr(v_cache_bits))


def attn_decode(qkv_new_bits, pos, heads, kv_heads, cap, scale, cos, sin, k_cache_bits,
                v_cache_bits, items=None, nthreads=None):
    """Decode outputs in float64: [n_seqs, heads*64], or [len(items), 64] for
    items = s*heads + h.  Caches must already hold row pos[s]."""
    lib = _load()
    q = np.ascontiguousarray(qkv_new_bits, np.uint16)
    pos = np.ascontiguousarray(pos, np.int32)
    n = len(pos)
    cos = np.ascontiguousarray(cos, np.float64)
    sin = np.ascontiguousarray(sin, np.float64)
    if items is None:
        out = np.zeros((n, heads * 64), np.float64)
        n_items, ip = n * heads, None
    else:
        ip = np.ascontiguousarray(items, np.int32)
        n_items = len(ip)
        out = np.zeros((n_items, 64), np.float64)
    rc = lib.kime_oracle_attn_decode(_ptr(q), _ptr(pos), n, heads, kv_heads, cap, float(scale),
                                     _ptr(cos), _ptr(sin), cos.shape[0], _ptr(k_cache_bits),
                                     _ptr(v_cache_bits), _ptr(ip), n_items, _ptr(out),
                                     _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def kv_append_varlen(qkv_bits, cu, pos, heads, kv_heads, cap, cos32, sin32, k_cache_bits, v_cache_bits):
    """Multi-token in-place append: row i of sequence s goes to cache row
    pos[s] + i of uint16 (bfloat16 bits) caches [n, kv_heads, cap, 64].
    Returns the number of sequences skipped for out-of-range positions."""
    lib = _load()
    q = np.ascontiguousarray(qkv_bits, np.uint16)
    cu = np.ascontiguousarray(cu, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    assert len(cu) == len(pos) + 1
    c = np.ascontiguousarray(cos32, np.float32)
    s = np.ascontiguousarray(sin32, np.float32)
    assert k_cache_bits.dtype == np.uint16 and k_cache_bits.flags.c_contiguous
    assert v_cache_bits.dtype == np.uint16 and v_cache_bits.flags.c_contiguous
    return lib.kime_oracle_kv_append_varlen(_ptr(q), _ptr(cu), _ptr(pos), len(pos), heads, kv_heads, cap,
                                            _ptr(c), _ptr(s), c.shape[0], _ptr(k_cache_bits),
                                            _ptr(v_cache_bits))


def attn_chunk(qkv_bits, cu, pos, heads, kv_heads, cap, scale, cos, sin, k_cache_bits, v_cache_bits,
               rows=None, row_heads=None, nthreads=None):
    """Chunked-prefill outputs in float64: row i of sequence s (position
    pos[s] + i) attends cache rows 0..pos[s]+i.  The caches must already hold
    the chunk (``kv_append_varlen``).  rows=None: [T, heads*64]; else the
    (row, head) items, [n, 64]."""
    lib = _load()
    q = np.ascontiguousarray(qkv_bits, np.uint16)
    cu = np.ascontiguousarray(cu, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    n = len(pos)
    assert len(cu) == n + 1
    cos = np.ascontiguousarray(cos, np.float64)
    sin = np.ascontiguousarray(sin, np.float64)
    if rows is None:
        T = int(cu[-1]) if n > 0 else 0
        out = np.zeros((T, heads * 64), np.float64)
        n_items, rp, hp = T * heads, None, None
    else:
        rp = np.ascontiguousarray(rows, np.int32)
        hp = np.ascontiguousarray(row_heads, np.int32)
        n_items = len(rp)
        out = np.zeros((n_items, 64), np.float64)
    rc = lib.kime_oracle_attn_chunk(_ptr(q), _ptr(cu), _ptr(pos), n, heads, kv_heads, cap, float(scale),
                                    _ptr(cos), _ptr(sin), cos.shape[0], _ptr(k_cache_bits),
                                    _ptr(v_cache_bits), _ptr(rp), _ptr(hp), n_items, _ptr(out),
                                    _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def qkv_proj(x_bits, w_bits, nthreads=None):
    """The QKV projection in float64: qkv [T, O] = x [T, K] . w [O, K]^T, with
    x and w given as bfloat16 bits (uint16); the weight is [out width, in width]."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, np.uint16)
    w = np.ascontiguousarray(w_bits, np.uint16)
    assert x.ndim == 2 and w.ndim == 2 and x.shape[1] == w.shape[1]
    out = np.zeros((x.shape[0], w.shape[0]), np.float64)
    rc = lib.kime_oracle_qkv_proj(_ptr(x), _ptr(w), x.shape[0], x.shape[1], w.shape[0], _ptr(out),
                                  _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def attn_varlen_proj(x_bits, w_bits, cu, heads, kv_heads, window, causal, scale, cos, sin, rows=None,
                     row_heads=None, nthreads=None):
    """Attention of a packed batch whose qkv rows are the projection of x:
    qkv_proj, then attn_varlen on the float64 rows (nothing rounded between)."""
    qkv = qkv_proj(x_bits, w_bits, nthreads)
    return attn_varlen(qkv, cu, heads, kv_heads, window, causal, scale, cos, sin, rows=rows,
                       row_heads=row_heads, nthreads=nthreads)
