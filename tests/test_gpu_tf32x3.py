"""GPU parity of the FP32 path on the tensor cores (KIME_F32_3XTF32: QK^T and PV
as three TF32 products each) against the FP64 oracle, through the C ABI: the
same FP32 contract (max abs error 1e-5) as the CUDA-core FP32 path, on the
same seeded inputs, plus the bitwise invariants that hold for any
implementation whose tiles are per sequence."""
import numpy as np
import pytest
import torch

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import cu_from_lengths, random_qkv, varlen_case

from parity_util import check_f32, gpu_tables, run_oracle_varlen, sample_items

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [0, 1, 2, 63, 64, 65, 127, 128, 129, 255]

CASES = [
    # lengths, H, Hkv, window, causal, scale
    (EDGE_LENGTHS, 2, 2, -1, False, 0.125),
    (EDGE_LENGTHS, 3, 1, -1, True, 0.125),
    (EDGE_LENGTHS, 2, 2, 64, False, 0.125),
    ([300, 129, 5], 3, 3, 1, True, 0.125),
    ([400, 1, 257], 9, 3, 65, True, 0.125),
    ([513, 200], 2, 1, 0, False, 0.125),
    ([250, 260], 4, 4, 300, False, 0.125),
    # scale 1 with the queries pre-scaled by 1/8, as the SmolLM2 prefill
    # workload stores them (unscaled N(0, 1) queries at scale 1 would give
    # logits eight times larger than any workload's)
    ([1500, 3, 700], 2, 2, -1, False, 1.0),
    ([1100, 0, 0, 90], 4, 2, 63, True, 0.125),
]


def run_3xtf32(qkv, cu, max_seqlen, H, Hkv, window, causal, scale, theta, rope_len=None, dev_status=None, out=None):
    dev = torch.device("cuda")
    c, s = gpu_tables(theta, rope_len or max(max_seqlen, 1))
    got = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), max_seqlen, H, Hkv, window, causal, scale, c, s,
                                out=out, dev_status=dev_status, precision="3xtf32")
    torch.cuda.synchronize()
    return got


def test_tiny_all_elements(cuda_lib):
    case = varlen_case("tiny")
    lay = case.layers[0]
    got = run_3xtf32(case.qkv, case.cu_seqlens, case.max_seqlen, case.heads, case.kv_heads, lay.window,
                     lay.causal, lay.scale, lay.theta)
    ref = run_oracle_varlen(case.qkv, case.cu_seqlens, case.heads, case.kv_heads, lay.window, lay.causal,
                            lay.scale, lay.theta, case.max_seqlen)
    assert got.dtype == torch.float32
    check_f32(got.cpu().numpy(), ref, "tiny 3xtf32")


@pytest.mark.parametrize("lengths,H,Hkv,window,causal,scale", CASES)
def test_small_all_elements(cuda_lib, lengths, H, Hkv, window, causal, scale):
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=61, q_scale=0.125 if scale == 1.0 else None)
    mx = max(lengths)
    got = run_3xtf32(qkv, cu, mx, H, Hkv, window, causal, scale, 1e4)
    ref = run_oracle_varlen(qkv, cu, H, Hkv, window, causal, scale, 1e4, mx)
    check_f32(got.cpu().numpy(), ref, f"3xtf32 {lengths} w{window} c{causal}")


def test_agrees_with_the_cuda_core_fp32_path(cuda_lib):
    # two FP32 implementations with different summation orders: each within
    # 1e-5 of the oracle, so within 2e-5 of each other
    lengths, H, Hkv = [700, 33, 129, 256], 4, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=62)
    dev = torch.device("cuda")
    c, s = gpu_tables(1e4, 700)
    a = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), 700, H, Hkv, 64, False, 0.125, c, s)
    b = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), 700, H, Hkv, 64, False, 0.125, c, s, precision="3xtf32")
    torch.cuda.synchronize()
    assert (a - b).abs().max().item() <= 2e-5


def test_modernbert_base_shapes_sampled(cuda_lib):
    # the ModernBERT-base workload's shapes (64 sequences of 32..512 tokens, 12
    # heads) in FP32, both layers, sampled rows against the oracle
    case = varlen_case("modernbert_base")
    qkv = case.qkv.float()
    for lay in case.layers:
        got = run_3xtf32(qkv, case.cu_seqlens, case.max_seqlen, case.heads, case.kv_heads, lay.window,
                         lay.causal, lay.scale, lay.theta)
        assert torch.isfinite(got).all()
        rows, hs = sample_items(case.cu_seqlens.numpy(), case.heads, 200, seed=63)
        ref = run_oracle_varlen(qkv, case.cu_seqlens, case.heads, case.kv_heads, lay.window, lay.causal,
                                lay.scale, lay.theta, case.max_seqlen, rows=rows, heads=hs)
        g = got.cpu().reshape(case.total, case.heads, 64)[torch.from_numpy(rows).long(), torch.from_numpy(hs).long()]
        check_f32(g.numpy(), ref, f"modernbert_base/{lay.name} 3xtf32")


def test_scale_fold_is_bitwise(cuda_lib):
    # q * 1/8 with scale 1 and q with scale 1/8 reach the same rotated, scaled
    # queries bit for bit (a power of two commutes with every rounding)
    lengths, H, Hkv = [300, 77], 6, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=64)
    folded = qkv.clone()
    folded[:, : H * 64] *= 0.125
    a = run_3xtf32(qkv, cu, 300, H, Hkv, -1, True, 0.125, 1e5)
    b = run_3xtf32(folded, cu, 300, H, Hkv, -1, True, 1.0, 1e5)
    assert torch.equal(a, b)


def test_window_at_least_length_is_bitwise_full(cuda_lib):
    lengths, H = [300, 77, 129], 3
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, H, torch.float32, 1.0, seed=65)
    full = run_3xtf32(qkv, cu, 300, H, H, -1, False, 0.125, 1e4)
    for w in (299, 300, 5000):
        assert torch.equal(run_3xtf32(qkv, cu, 300, H, H, w, False, 0.125, 1e4), full)


def test_packing_order_does_not_change_a_sequence_bitwise(cuda_lib):
    # a sequence's rows sit elsewhere in another packing (and its last key
    # half reaches into other neighbours); its results do not move
    lengths, H, Hkv = [333, 10, 129, 512], 6, 3
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=66)
    cu = cu_from_lengths(lengths)
    order = [2, 0, 3, 1]
    pieces = [qkv[int(cu[s]):int(cu[s + 1])] for s in range(4)]
    qkv2 = torch.cat([pieces[s] for s in order])
    cu2 = cu_from_lengths([lengths[s] for s in order])
    for window, causal in [(-1, False), (64, False), (-1, True)]:
        a = run_3xtf32(qkv, cu, 512, H, Hkv, window, causal, 0.125, 1e4).cpu()
        b = run_3xtf32(qkv2, cu2, 512, H, Hkv, window, causal, 0.125, 1e4).cpu()
        for k, s in enumerate(order):
            assert torch.equal(a[int(cu[s]):int(cu[s + 1])], b[int(cu2[k]):int(cu2[k + 1])])


def test_single_keys_and_window_zero_return_v(cuda_lib):
    # softmax over one visible key is exactly 1 (p_hi = 1, p_lo = 0), so the
    # output is v_hi + v_lo with v_lo truncated to TF32 by the tensor core:
    # v to within 2^-20 |v| (the truncation drops at most the last two of
    # v_lo's 13 significant bits)
    lengths, H, Hkv = [1, 5, 1, 130], 4, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=67)
    got = run_3xtf32(qkv, cu, 130, H, Hkv, 0, False, 0.125, 1e4).cpu().reshape(-1, H, 64).double()
    v = qkv[:, (H + Hkv) * 64:].reshape(-1, Hkv, 64).double()
    for h in range(H):
        want = v[:, h // (H // Hkv)]
        assert torch.all((got[:, h] - want).abs() <= 2.0 ** -20 * want.abs())


def test_device_status_flags_bad_cu_and_skips(cuda_lib):
    dev = torch.device("cuda")
    lengths, H = [100, 50, 30], 2
    qkv = random_qkv(lengths, H, H, torch.float32, 1.0, seed=68)
    # the last sequence ends past the 180 rows of qkv / out: it must be skipped
    cu = torch.tensor([0, 100, 150, 200], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full((180, H * 64), 7.0, dtype=torch.float32, device=dev)
    run_3xtf32(qkv, cu, 100, H, H, -1, False, 0.125, 1e4, rope_len=200, dev_status=st, out=out)
    assert int(st.item()) & kime.DEV_BAD_CU
    o = out.cpu()
    assert torch.all(o[150:180] == 7.0) and not torch.all(o[:150] == 7.0)
    ref = run_3xtf32(qkv[:150], cu_from_lengths([100, 50]), 100, H, H, -1, False, 0.125, 1e4, rope_len=200).cpu()
    assert torch.equal(o[:150], ref)


def test_workspace_too_small_and_dtype_errors_raise(cuda_lib):
    dev = torch.device("cuda")
    lengths, H = [40, 9], 2
    qkv = random_qkv(lengths, H, H, torch.float32, 1.0, seed=69).to(dev)
    cu = cu_from_lengths(lengths).to(dev)
    c, s = gpu_tables(1e4, 64)
    small = torch.empty(kime.kime_attn_workspace_bytes(4, 2, 49, H, H) - 8, dtype=torch.uint8, device=dev)
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 40, H, H, -1, False, 0.125, c, s, workspace=small, precision="3xtf32")
    with pytest.raises(TypeError):
        kime.kime_attn_varlen(qkv.bfloat16(), cu, 40, H, H, -1, False, 0.125, c, s, precision="3xtf32")


def test_replays_from_a_cuda_graph(cuda_lib):
    # the scheduler and the attention kernel are both on the given stream and
    # allocate nothing: one capture, replayed on new inputs
    dev = torch.device("cuda")
    lengths, H, Hkv = [700, 1, 129, 300], 4, 2
    cu = cu_from_lengths(lengths).to(dev)
    T, n = sum(lengths), len(lengths)
    c, s = gpu_tables(1e4, 700)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=70).to(dev)
    ws = torch.empty(kime.kime_attn_workspace_bytes(4, n, T, H, Hkv), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H * 64), dtype=torch.float32, device=dev)
    call = lambda o: kime.kime_attn_varlen(qkv, cu, 700, H, Hkv, -1, True, 0.125, c, s, out=o, workspace=ws,
                                           precision="3xtf32")
    call(out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out)
    for seed in (71, 72):
        qkv.copy_(random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=seed).to(dev))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        want = call(torch.empty_like(out))
        torch.cuda.synchronize()
        assert torch.equal(out, want), seed
