"""kime_attn_varlen_noalloc: the entry point for callers that cannot allocate
device memory at call time (its scratch is a fixed array inside the library).
Its output must equal kime_attn_varlen's -- the entry point that takes a
caller-provided workspace -- given the workspace size that makes that entry
point take the same kernels (the no-alloc entry hands the library its whole
array, so prepared rows are used exactly when they fit in it).  Calls come in
pairs of different shapes, which also shows that what one call leaves in the
shared scratch does not disturb the next.  This file is collected last on
purpose."""
import ctypes

import pytest
import torch

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import cu_from_lengths, random_qkv

from parity_util import gpu_tables

pytestmark = pytest.mark.gpu


def _ref_workspace(n, T, H, Hkv, dtype, dev):
    """The workspace kime_attn_varlen gets in the comparison: of the size that
    selects the kernels the no-alloc entry takes with its built-in array."""
    if dtype == torch.bfloat16:
        prep = kime.kime_attn_workspace_bytes(3, n, T, H, Hkv)
        nbytes = prep if prep <= kime.NOALLOC_SCRATCH_BYTES else kime.kime_attn_workspace_bytes(0, n, T)
    else:
        nbytes = kime.kime_attn_workspace_bytes(0, n, T)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)


def _pair(lengths, H, Hkv, dtype, window, causal, scale, seed):
    dev = torch.device("cuda")
    qkv = random_qkv(lengths, H, Hkv, dtype, 1.5, seed=seed).to(dev)
    cu = cu_from_lengths(lengths).to(dev)
    mx = max(lengths)
    c, s = gpu_tables(1e4, mx)
    ws = _ref_workspace(len(lengths), qkv.shape[0], H, Hkv, dtype, dev)
    ref = kime.kime_attn_varlen(qkv, cu, mx, H, Hkv, window, causal, scale, c, s, workspace=ws)
    got = kime.kime_attn_varlen_noalloc(qkv, cu, mx, H, Hkv, window, causal, scale, c, s)
    torch.cuda.synchronize()
    return got.cpu(), ref.cpu()


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cuda_lib):
    # BF16 too large for prepared rows in the array (the kernel that rotates
    # in place), then causal GQA with other shapes, then a batch whose
    # prepared rows fit (the prepared-rows kernel), then FP32
    cases = [
        ([300, 129, 1, 512, 77], 4, 4, torch.bfloat16, 64, False, 0.125, 31),
        ([1142, 700], 9, 3, torch.bfloat16, -1, True, 0.125, 32),
        ([7, 13], 2, 2, torch.bfloat16, -1, False, 0.125, 34),
        ([200, 3], 3, 1, torch.bfloat16, 1, True, 0.125, 35),
        ([7, 13], 2, 2, torch.float32, -1, False, 0.125, 33),
    ]
    n_prep = 0
    for lengths, H, Hkv, dtype, window, causal, scale, seed in cases:
        T = sum(lengths)
        if dtype == torch.bfloat16 and kime.kime_attn_workspace_bytes(3, len(lengths), T, H, Hkv) <= \
                kime.NOALLOC_SCRATCH_BYTES:
            n_prep += 1
        got, ref = _pair(lengths, H, Hkv, dtype, window, causal, scale, seed)
        assert torch.equal(got, ref), (lengths, H, Hkv, dtype, window, causal)
    assert n_prep == 2  # the prepared-rows path through the array ran twice


def test_noalloc_3xtf32_through_the_c_abi(cuda_lib):
    # the Python wrapper passes only qkv's own dtype; the C entry also takes
    # KIME_F32_3XTF32 (whose scratch is the scheduler's alone)
    dev = torch.device("cuda")
    lib = kime.load_library()
    for lengths, H, Hkv, window, causal, seed in [([7, 13], 2, 2, -1, False, 36), ([40, 9], 3, 1, 4, True, 37)]:
        T, n = sum(lengths), len(lengths)
        assert kime.kime_attn_workspace_bytes(4, n, T, H, Hkv) <= kime.NOALLOC_SCRATCH_BYTES
        qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=seed).to(dev)
        cu = cu_from_lengths(lengths).to(dev)
        mx = max(lengths)
        c, s = gpu_tables(1e4, mx)
        ref = kime.kime_attn_varlen(qkv, cu, mx, H, Hkv, window, causal, 0.125, c, s, precision="3xtf32")
        got = torch.empty_like(ref)
        stream = torch.cuda.current_stream(dev)
        rc = lib.kime_attn_varlen_noalloc(
            ctypes.c_void_p(qkv.data_ptr()), kime.KIME_F32_3XTF32, ctypes.c_void_p(cu.data_ptr()), n, T, mx, H,
            Hkv, 64, window, int(causal), 0.125, ctypes.c_void_p(c.data_ptr()), ctypes.c_void_p(s.data_ptr()),
            c.shape[0], ctypes.c_void_p(got.data_ptr()), None, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_rejects_a_batch_beyond_its_scratch(cuda_lib):
    dev = torch.device("cuda")
    # enough sequences that the scheduler's scratch alone passes the array by a clear margin
    n = 1
    while kime.kime_attn_workspace_bytes(0, n, 0) <= kime.NOALLOC_SCRATCH_BYTES * 5 // 4:
        n *= 2
    assert kime.kime_attn_workspace_bytes(0, n, 0) > kime.NOALLOC_SCRATCH_BYTES
    cu = torch.zeros(n + 1, dtype=torch.int32, device=dev)
    qkv = torch.zeros((1, 64 * 3), dtype=torch.bfloat16, device=dev)
    c, s = gpu_tables(1e4, 4)
    with pytest.raises(kime.KimeError) as e:
        kime.kime_attn_varlen_noalloc(qkv, cu, 1, 1, 1, -1, False, 0.125, c, s)
    assert e.value.status == -2  # KIME_ERANGE
