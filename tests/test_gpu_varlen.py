"""GPU parity of kime_attn_varlen (scheduler, FP32 SIMT path, BF16 tcgen05 path)
against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tiles as otiles
import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import cu_from_lengths, random_qkv, varlen_case

from parity_util import (check_bf16, check_f32, gpu_tables, run_gpu_varlen, run_oracle_varlen,
                         sample_items)

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [0, 1, 2, 63, 64, 65, 127, 128, 129, 255]
WINDOWS = [-1, 0, 1, 63, 64, 65, 300]


def codes_from_gpu(tiles):
    out = {}
    for row in tiles.cpu().numpy():
        s, qt, kb, ke, fb, fe, row0, L = [int(v) for v in row]
        nk = -(-L // 128)
        codes = np.zeros(nk, np.int8)
        codes[kb:ke] = 1
        codes[fb:fe] = 2
        out[(s, qt)] = codes
    return out


def assert_tiles_equal(cu, total, max_seqlen, causal, window):
    dev = torch.device("cuda")
    tiles = kime.kime_attn_debug_tiles(cu.to(dev), total, max_seqlen, window, causal)
    got = codes_from_gpu(tiles)
    want = otiles.classify(cu.numpy(), causal, window)
    assert set(got) == set(want)
    for k in want:
        assert np.array_equal(got[k], want[k]), (k, got[k], want[k])
    # longest-first order: the number of visited key tiles never increases
    cost = (tiles[:, 3] - tiles[:, 2]).cpu().numpy()
    assert np.all(np.diff(np.minimum(cost, 255)) <= 0)


def test_rope_tables_match_the_oracle_bitwise(cuda_lib):
    for theta in (1e4, 1e5, 1.6e5):
        c, s = kime.kime_rope_tables(theta, 8192)
        oc, os_ = oracle.rope_tables_f32(theta, 8192)
        assert np.array_equal(c.numpy(), oc) and np.array_equal(s.numpy(), os_)


@pytest.mark.parametrize("causal", [False, True])
def test_schedule_small_shapes_bit_exact(cuda_lib, causal):
    cu = cu_from_lengths(EDGE_LENGTHS + [700, 3, 1000])
    total = int(cu[-1])
    for w in WINDOWS + [127, 128, 2000]:
        assert_tiles_equal(cu, total, 1000, causal, w)
    # few long sequences (the scheduler then gives each sequence a warp)
    cu = cu_from_lengths([3000, 1, 5000, 4097, 0])
    for w in WINDOWS + [2000, 6000]:
        assert_tiles_equal(cu, int(cu[-1]), 5000, causal, w)


@pytest.mark.parametrize("name", ["modernbert_base", "modernbert_large", "smollm2_prefill"])
def test_schedule_workloads_bit_exact(cuda_lib, name):
    case = varlen_case(name) if name != "modernbert_large" else None
    if case is None:  # lengths only; values are not needed here
        g = torch.Generator().manual_seed(3)
        lengths = [int(v) for v in torch.randint(1024, 8193, (8,), generator=g)]
        cu = cu_from_lengths(lengths)
        layers = [(64, False), (-1, False)]
        total, mx = int(cu[-1]), max(lengths)
    else:
        cu, total, mx = case.cu_seqlens, case.total, case.max_seqlen
        layers = [(l.window, l.causal) for l in case.layers]
    for w, causal in layers:
        assert_tiles_equal(cu, total, mx, causal, w)


def test_varlen_f32_tiny_all_elements(cuda_lib):
    case = varlen_case("tiny")
    lay = case.layers[0]
    got = run_gpu_varlen(case.qkv, case.cu_seqlens, case.max_seqlen, case.heads, case.kv_heads, lay.window,
                         lay.causal, lay.scale, lay.theta)
    ref = run_oracle_varlen(case.qkv, case.cu_seqlens, case.heads, case.kv_heads, lay.window, lay.causal,
                            lay.scale, lay.theta, case.max_seqlen)
    check_f32(got.cpu().numpy(), ref, "tiny fp32")


SMALL = [
    # lengths, H, Hkv, window, causal, scale
    (EDGE_LENGTHS, 2, 2, -1, False, 0.125),
    (EDGE_LENGTHS, 3, 1, -1, True, 0.125),
    (EDGE_LENGTHS, 2, 2, 64, False, 0.125),
    ([300, 129, 5], 3, 3, 1, True, 0.125),
    ([400, 1, 257], 9, 3, 65, True, 0.125),
    ([513, 200], 2, 1, 0, False, 0.125),
    ([250, 260], 4, 4, 300, False, 0.125),
    # long sequences with window 64: units past the first take their key tiles
    # on a grid starting at their first visible key (not 128-aligned)
    ([1100, 700], 4, 2, 64, False, 0.125),
]


@pytest.mark.parametrize("out_dtype,u", [(torch.float16, 2.0 ** -11), (torch.bfloat16, 2.0 ** -8)])
def test_varlen_f32_qkv_16bit_out(cuda_lib, out_dtype, u):
    # kime-cuda's mixed precision (FP32 qkv, 16-bit attention output): the
    # output is the FP32 path's result rounded once to nearest even, bit for
    # bit, so against the oracle it is within 1e-5 plus half an ulp
    lengths, H, Hkv, window, causal = [300, 129, 5, 1], 3, 1, 64, True
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=41)
    dev = torch.device("cuda")
    c, s = gpu_tables(1e4, max(lengths))
    f32 = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), max(lengths), H, Hkv, window, causal, 0.125, c, s)
    o16 = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), max(lengths), H, Hkv, window, causal, 0.125, c, s,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert o16.dtype == out_dtype
    assert torch.equal(o16.view(torch.int16), f32.to(out_dtype).view(torch.int16))
    ref = run_oracle_varlen(qkv, cu, H, Hkv, window, causal, 0.125, 1e4, max(lengths))
    got = o16.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-5 * (1 + u) + u * np.abs(ref))


@pytest.mark.parametrize("lengths,H,Hkv,window,causal,scale", SMALL)
def test_varlen_f32_small_all_elements(cuda_lib, lengths, H, Hkv, window, causal, scale):
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.float32, 1.0, seed=11)
    mx = max(lengths)
    got = run_gpu_varlen(qkv, cu, mx, H, Hkv, window, causal, scale, 1e4)
    ref = run_oracle_varlen(qkv, cu, H, Hkv, window, causal, scale, 1e4, mx)
    check_f32(got.cpu().numpy(), ref, f"fp32 {lengths} w{window} c{causal}")


@pytest.mark.parametrize("lengths,H,Hkv,window,causal,scale", SMALL)
def test_varlen_bf16_small_all_elements(cuda_lib, lengths, H, Hkv, window, causal, scale):
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=12)
    mx = max(lengths)
    got = run_gpu_varlen(qkv, cu, mx, H, Hkv, window, causal, scale, 1e4)
    ref = run_oracle_varlen(qkv, cu, H, Hkv, window, causal, scale, 1e4, mx)
    check_bf16(got.float().cpu().numpy(), ref, f"bf16 {lengths} w{window} c{causal}")


def test_varlen_bf16_window_zero_and_single_tokens_return_v_exactly(cuda_lib):
    lengths, H, Hkv = [1, 200, 1, 130], 4, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=13)
    v = qkv[:, (H + Hkv) * 64:].reshape(-1, Hkv, 64)
    out = run_gpu_varlen(qkv, cu, 200, H, Hkv, 0, False, 0.125, 1e4).cpu().reshape(-1, H, 64)
    for h in range(H):
        assert torch.equal(out[:, h], v[:, h // (H // Hkv)])
    full = run_gpu_varlen(qkv, cu, 200, H, Hkv, -1, False, 0.125, 1e4).cpu().reshape(-1, H, 64)
    for r in (0, 201):  # the length-1 sequences
        for h in range(H):
            assert torch.equal(full[r, h], v[r, h // (H // Hkv)])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_scale_fold_is_bitwise_on_gpu(cuda_lib, dtype):
    lengths, H, Hkv = [300, 77], 6, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, dtype, 1.0, seed=14)
    folded = qkv.clone()
    folded[:, : H * 64] = (folded[:, : H * 64].float() * 0.125).to(dtype)
    a = run_gpu_varlen(qkv, cu, 300, H, Hkv, -1, True, 0.125, 1e5)
    b = run_gpu_varlen(folded, cu, 300, H, Hkv, -1, True, 1.0, 1e5)
    assert torch.equal(a, b)


def test_window_at_least_length_is_bitwise_full_on_gpu(cuda_lib):
    lengths, H = [300, 77, 129], 3
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, H, torch.bfloat16, 1.5, seed=15)
    full = run_gpu_varlen(qkv, cu, 300, H, H, -1, False, 0.125, 1e4)
    for w in (299, 300, 5000):
        assert torch.equal(run_gpu_varlen(qkv, cu, 300, H, H, w, False, 0.125, 1e4), full)


def test_packing_order_does_not_change_a_sequence_bitwise(cuda_lib):
    lengths, H, Hkv = [333, 10, 129, 512], 6, 3
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=16)
    cu = cu_from_lengths(lengths)
    order = [2, 0, 3, 1]
    pieces = [qkv[int(cu[s]):int(cu[s + 1])] for s in range(4)]
    qkv2 = torch.cat([pieces[s] for s in order])
    cu2 = cu_from_lengths([lengths[s] for s in order])
    for window, causal in [(-1, False), (64, False), (-1, True)]:
        a = run_gpu_varlen(qkv, cu, 512, H, Hkv, window, causal, 0.125, 1e4).cpu()
        b = run_gpu_varlen(qkv2, cu2, 512, H, Hkv, window, causal, 0.125, 1e4).cpu()
        for k, s in enumerate(order):
            assert torch.equal(a[int(cu[s]):int(cu[s + 1])], b[int(cu2[k]):int(cu2[k + 1])])


@pytest.mark.parametrize("name", ["modernbert_base", "modernbert_large", "smollm2_prefill"])
def test_workloads_full_size_sampled(cuda_lib, name):
    case = varlen_case(name, device="cuda")
    qkv_cpu = case.qkv.cpu()
    for lay in case.layers:
        got = run_gpu_varlen(case.qkv, case.cu_seqlens, case.max_seqlen, case.heads, case.kv_heads,
                             lay.window, lay.causal, lay.scale, lay.theta)
        assert torch.isfinite(got.float()).all()
        rows, hs = sample_items(case.cu_seqlens.numpy(), case.heads, 400, seed=len(name))
        ref = run_oracle_varlen(qkv_cpu, case.cu_seqlens, case.heads, case.kv_heads, lay.window, lay.causal,
                                lay.scale, lay.theta, case.max_seqlen, rows=rows, heads=hs)
        g = got.float().cpu().reshape(case.total, case.heads, 64)[torch.from_numpy(rows).long(),
                                                                   torch.from_numpy(hs).long()]
        check_bf16(g.numpy(), ref, f"{name}/{lay.name}")


PREP_CASES = [
    ([1500, 700, 1, 129, 2100], 4, 2, -1, False),
    ([1500, 700, 1, 129, 2100], 4, 2, -1, True),
    ([1500, 700, 1, 129, 2100], 4, 2, 600, False),
    ([1, 2, 63, 64, 65, 127, 128, 129, 255, 300, 0, 513], 3, 1, 64, False),
    ([1, 2, 63, 64, 65, 127, 128, 129, 255, 300, 0, 513], 3, 3, 0, False),
    ([1, 2, 63, 64, 65, 127, 128, 129, 255, 300, 0, 513], 6, 2, -1, True),
]


@pytest.mark.parametrize("lengths,H,Hkv,window,causal", PREP_CASES)
def test_prepared_rows_and_fused_paths_match_the_oracle(cuda_lib, lengths, H, Hkv, window, causal):
    # With a workspace of op 3 size the qkv rows are prepared once (RoPE, the
    # query scale, f16) and the attention kernel over prepared rows runs; with
    # the minimal workspace (op 0) the kernel
    # that rotates queries and key tiles itself runs.  Both are checked
    # against the oracle on the same sampled rows.
    dev = torch.device("cuda")
    qkv_cpu = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=31)
    qkv = qkv_cpu.to(dev)
    cu = cu_from_lengths(lengths)
    T, n, mx = qkv.shape[0], len(lengths), max(lengths)
    assert kime.kime_attn_workspace_bytes(3, n, T, H, Hkv) > kime.kime_attn_workspace_bytes(0, n, T)
    c, s = gpu_tables(1e4, mx)
    outs = []
    for op in (0, 3):
        ws = torch.empty(kime.kime_attn_workspace_bytes(op, n, T, H, Hkv), dtype=torch.uint8, device=dev)
        outs.append(kime.kime_attn_varlen(qkv, cu.to(dev), mx, H, Hkv, window, causal, 0.125, c, s, workspace=ws))
    torch.cuda.synchronize()
    rows, hs = sample_items(cu.numpy(), H, 300, seed=5)
    ref = run_oracle_varlen(qkv_cpu, cu, H, Hkv, window, causal, 0.125, 1e4, mx, rows=rows, heads=hs)
    for op, o in zip((0, 3), outs):
        g = o.float().cpu().reshape(T, H, 64)[torch.from_numpy(rows).long(), torch.from_numpy(hs).long()]
        check_bf16(g.numpy(), ref, f"op {op} {lengths} w{window} c{causal}")


# Sequences with an odd number of query tiles end in a unit of one tile (1-,
# 3- and 9-tile sequences here, of several costs), next to units of two.
ODD_TILES = [300, 290, 260, 1100, 1150, 100, 120, 128, 50]
ODD_CASES = [
    (ODD_TILES, 4, 2, -1, False),
    (ODD_TILES, 4, 2, -1, True),
    (ODD_TILES, 4, 4, 64, False),
    (ODD_TILES, 6, 2, 200, True),
]


@pytest.mark.parametrize("lengths,H,Hkv,window,causal", ODD_CASES)
def test_odd_tile_counts_match_the_oracle_everywhere(cuda_lib, lengths, H, Hkv, window, causal):
    dev = torch.device("cuda")
    qkv_cpu = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=41)
    cu = cu_from_lengths(lengths)
    T, n, mx = qkv_cpu.shape[0], len(lengths), max(lengths)
    c, s = gpu_tables(1e4, mx)
    ws = torch.empty(kime.kime_attn_workspace_bytes(3, n, T, H, Hkv), dtype=torch.uint8, device=dev)
    out = kime.kime_attn_varlen(qkv_cpu.to(dev), cu.to(dev), mx, H, Hkv, window, causal, 0.125, c, s, workspace=ws)
    torch.cuda.synchronize()
    ref = run_oracle_varlen(qkv_cpu, cu, H, Hkv, window, causal, 0.125, 1e4, mx)
    check_bf16(out.float().cpu().numpy().reshape(ref.shape), ref, f"odd tile counts w{window} c{causal}")


@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (False, 200)])
def test_both_epilogue_stores_give_the_same_bits(cuda_lib, causal, window):
    # The kernel over prepared rows has two epilogues: stores coalesced
    # through a four-lane transpose (batches of short sequences) or one row
    # per thread (long ones).  A 300-token sequence alone takes the first,
    # packed with a 7,000-token one the second; its rows match bit for bit.
    dev = torch.device("cuda")
    H, Hkv = 4, 2
    both = random_qkv([300, 7000], H, Hkv, torch.bfloat16, 1.5, seed=45)
    outs = []
    for lengths, qkv in (([300], both[:300]), ([300, 7000], both)):
        cu = cu_from_lengths(lengths)
        T, n, mx = qkv.shape[0], len(lengths), max(lengths)
        c, s = gpu_tables(1e4, mx)
        ws = torch.empty(kime.kime_attn_workspace_bytes(3, n, T, H, Hkv), dtype=torch.uint8, device=dev)
        outs.append(kime.kime_attn_varlen(qkv.contiguous().to(dev), cu.to(dev), mx, H, Hkv, window, causal, 0.125,
                                          c, s, workspace=ws))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1][:300])


def test_device_status_flags_bad_cu_and_skips(cuda_lib):
    dev = torch.device("cuda")
    lengths, H = [100, 50, 30], 2
    qkv = random_qkv(lengths, H, H, torch.bfloat16, 1.0, seed=17)
    # the last sequence ends past the 180 rows of qkv / out: it must be skipped
    cu = torch.tensor([0, 100, 150, 200], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    c, s = gpu_tables(1e4, 200)
    out = torch.full((180, H * 64), 7.0, dtype=torch.bfloat16, device=dev)
    kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), 100, H, H, -1, False, 0.125, c, s, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kime.DEV_BAD_CU
    o = out.cpu().float()
    assert torch.all(o[150:180] == 7.0) and not torch.all(o[:150] == 7.0)
    ref = run_gpu_varlen(qkv[:150], cu_from_lengths([100, 50]), 100, H, H, -1, False, 0.125, 1e4).cpu().float()
    assert torch.equal(o[:150], ref)
    # too long for max_seqlen: skipped and flagged
    st.zero_()
    cu = cu_from_lengths(lengths).to(dev)
    out.fill_(7.0)
    kime.kime_attn_varlen(qkv.to(dev), cu, 60, H, H, -1, False, 0.125, c, s, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kime.DEV_SEQ_TOO_LONG
    o = out.cpu().float()
    assert torch.all(o[:100] == 7.0) and not torch.all(o[100:150] == 7.0)


def test_host_argument_errors_raise(cuda_lib):
    dev = torch.device("cuda")
    qkv = torch.zeros((10, 64 * 6), dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, 10], dtype=torch.int32, device=dev)
    c, s = gpu_tables(1e4, 16)
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 10, 2, 2, -2, False, 0.125, c, s)   # window < -1
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 10, 3, 2, -1, False, 0.125, c, s)   # heads % kv_heads
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 17, 2, 2, -1, False, 0.125, c, s)   # max_seqlen > rope_len
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 10, 2, 2, -1, False, 0.0, c, s)     # scale
    with pytest.raises(kime.KimeError):
        kime.kime_attn_varlen(qkv, cu, 10, 2, 2, -1, False, 0.125, c, s,
                              workspace=torch.empty(8, dtype=torch.uint8, device=dev))
    # empty batch is fine and launches nothing
    e = kime.kime_attn_varlen(qkv[:0], torch.zeros(1, dtype=torch.int32, device=dev), 0, 2, 2, -1, False,
                              0.125, c, s)
    assert e.shape[0] == 0


def test_narrow_window_over_long_sequences_meets_the_contract_with_either_workspace(cuda_lib):
    # A window of 64 over long sequences, through the minimal workspace (the
    # kernel that rotates its own tiles, every tile on its partial path) and
    # the row-preparing one (prepared rows, every tile on the partial path):
    # both meet the BF16 contract against the oracle on sampled rows.
    dev = torch.device("cuda")
    lengths, H, Hkv = [1500, 1100, 1300], 4, 2
    cu = cu_from_lengths(lengths)
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=14).to(dev)
    T, n, mx = sum(lengths), len(lengths), max(lengths)
    c, s = gpu_tables(1e4, mx)
    outs = {}
    for op in (0, 3):
        ws = torch.empty(kime.kime_attn_workspace_bytes(op, n, T, H, Hkv), dtype=torch.uint8, device=dev)
        outs[op] = kime.kime_attn_varlen(qkv, cu.to(dev), mx, H, Hkv, 64, False, 0.125, c, s, workspace=ws)
    torch.cuda.synchronize()
    rows, hs = sample_items(cu.numpy(), H, 200, seed=15)
    ref = run_oracle_varlen(qkv.cpu(), cu, H, Hkv, 64, False, 0.125, 1e4, mx, rows=rows, heads=hs)
    for op in (0, 3):
        g = outs[op].float().cpu().reshape(T, H, 64)[torch.from_numpy(rows).long(), torch.from_numpy(hs).long()]
        check_bf16(g.numpy(), ref, f"window 64, long sequences, op {op}")
