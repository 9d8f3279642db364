"""kime_attn_varlen_noalloc: the entry point for callers that cannot allocate
device memory at call time (its scratch is a fixed array inside the library).
Its output must match kime_attn_varlen's -- the entry point that takes a
caller-provided workspace -- on two calls in a row, which also shows that the
shared scratch left behind by one call does not disturb the next.  This file
is collected last on purpose."""
import pytest
import torch

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import cu_from_lengths, random_qkv

from parity_util import check_bf16, check_f32, gpu_tables

pytestmark = pytest.mark.gpu


def _pair(lengths, H, Hkv, dtype, window, causal, scale, seed):
    dev = torch.device("cuda")
    qkv = random_qkv(lengths, H, Hkv, dtype, 1.5, seed=seed).to(dev)
    cu = cu_from_lengths(lengths).to(dev)
    mx = max(lengths)
    c, s = gpu_tables(1e4, mx)
    ref = kime.kime_attn_varlen(qkv, cu, mx, H, Hkv, window, causal, scale, c, s)
    got = kime.kime_attn_varlen_noalloc(qkv, cu, mx, H, Hkv, window, causal, scale, c, s)
    torch.cuda.synchronize()
    return got.float().cpu().numpy(), ref.float().cpu().numpy()


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cuda_lib):
    # call 1: BF16, many short sequences, windowed; call 2: BF16 causal GQA with
    # longer sequences, so the second call's schedule differs from the first's.
    got, ref = _pair([300, 129, 1, 512, 77], 4, 4, torch.bfloat16, 64, False, 0.125, seed=31)
    check_bf16(got, ref, "noalloc call 1")
    got, ref = _pair([1142, 700], 9, 3, torch.bfloat16, -1, True, 0.125, seed=32)
    check_bf16(got, ref, "noalloc call 2")
    got, ref = _pair([7, 13], 2, 2, torch.float32, -1, False, 0.125, seed=33)
    check_f32(got, ref, "noalloc fp32")


def test_noalloc_rejects_a_batch_beyond_its_scratch(cuda_lib):
    dev = torch.device("cuda")
    n = kime.NOALLOC_SCRATCH_BYTES // 64 + 10  # more sequences than the scratch can schedule
    cu = torch.zeros(n + 1, dtype=torch.int32, device=dev)
    qkv = torch.zeros((1, 64 * 3), dtype=torch.bfloat16, device=dev)
    c, s = gpu_tables(1e4, 4)
    with pytest.raises(kime.KimeError) as e:
        kime.kime_attn_varlen_noalloc(qkv, cu, 1, 1, 1, -1, False, 0.125, c, s)
    assert e.value.status == -2  # KIME_ERANGE
