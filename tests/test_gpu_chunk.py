"""GPU parity of chunked prefill against the KV cache (kime_kv_append_varlen,
kime_attn_chunk, kime_chunk_step) and of its scheduler, against the FP64
oracle, through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_kime_gb300 as kime
from oracle import tiles as otiles
from packed_varlen_attention_kime_gb300.inputs import bf16_bits, chunk_case

from parity_util import check_bf16, gpu_tables, oracle_tables, sample_items

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0  # a quiet NaN bit pattern


def poison_unused_rows(case):
    """Cache rows at and past pos[s] + L are never attended: fill them with NaN
    so that a kernel reading one (or not zeroing it) shows."""
    for s, L in enumerate(case.lengths):
        end = int(case.pos[s]) + L
        case.k_cache[s, :, end:].view(torch.int16).fill_(NAN_BF16)
        case.v_cache[s, :, end:].view(torch.int16).fill_(NAN_BF16)


def gpu_chunk(case, mode="step", dev_status=None, ws_op=None):
    """mode: 'step' (kime_chunk_step), 'split' (append then attend).  ws_op:
    the workspace size (2: the kernel that converts its own tiles, 5: the one
    over prepared rows); None: the binding's default."""
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.cap)
    qkv, cu, pos = case.qkv.to(dev), case.cu_seqlens.to(dev), case.pos.to(dev)
    kc, vc = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    args = (qkv, cu, pos, max(case.max_seqlen, 1), case.heads, case.kv_heads, kc, vc, case.scale, c, s)
    ws = None
    if ws_op is not None:
        nb = kime.kime_attn_workspace_bytes(ws_op, len(case.lengths), case.total, case.heads, case.kv_heads, case.cap)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
    if mode == "step":
        out = kime.kime_chunk_step(*args, workspace=ws, dev_status=dev_status)
    else:
        kime.kime_kv_append_varlen(qkv, cu, pos, case.heads, case.kv_heads, kc, vc, c, s, dev_status=dev_status)
        out = kime.kime_attn_chunk(*args, workspace=ws, dev_status=dev_status)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_chunk(case, rows=None, heads=None):
    qb = bf16_bits(case.qkv)
    cu = case.cu_seqlens.numpy()
    pos = case.pos.numpy()
    kb = bf16_bits(case.k_cache).copy()
    vb = bf16_bits(case.v_cache).copy()
    c32, s32 = oracle.rope_tables_f32(case.theta, case.cap)
    assert oracle.kv_append_varlen(qb, cu, pos, case.heads, case.kv_heads, case.cap, c32, s32, kb, vb) == 0
    c, s = oracle_tables(case.theta, case.cap)
    out = oracle.attn_chunk(qb, cu, pos, case.heads, case.kv_heads, case.cap, case.scale, c, s, kb, vb,
                            rows=rows, row_heads=heads)
    return out, kb, vb


# ---- scheduler ------------------------------------------------------------------

@pytest.mark.parametrize("lengths,pos", [
    ([1, 5, 128, 129, 300, 0, 257], [0, 200, 128, 126, 1000, 7, 383]),
    ([1000, 1, 1, 640], [0, 0, 4095, 3]),
])
def test_chunk_schedule_is_bit_exact(cuda_lib, lengths, pos):
    cu = kime_cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    total, cap = int(cu[-1]), 5000
    tiles = kime.kime_attn_debug_tiles_chunk(kime_cu.cuda(), torch.tensor(pos, dtype=torch.int32).cuda(), total,
                                             max(lengths), cap, cap).cpu().numpy()
    want = otiles.classify(cu.numpy(), True, -1, pos=pos)
    assert len(tiles) == len(want)
    got = {}
    for s, qt, kb, ke, fb, fe, row0, L in tiles:
        assert row0 == cu[s] and L == lengths[s]
        codes = np.zeros(len(want[(s, qt)]), np.int8)
        codes[kb:ke] = 1
        codes[fb:fe] = 2
        got[(s, qt)] = codes
    for key, codes in want.items():
        assert np.array_equal(got[key], codes), key


# ---- append + attention -------------------------------------------------------------

@pytest.mark.parametrize("mode", ["split", "step"])
def test_chunk_small_all_outputs(cuda_lib, mode):
    # tile edges in both the chunk length and the cache offset; an empty chunk;
    # a chunk that ends at the last cache row
    lengths = [1, 5, 128, 129, 300, 0, 257, 64]
    pos = [0, 200, 128, 126, 1000, 7, 383, 1536]
    case = chunk_case(lengths=lengths, pos=pos, cap=1600, seed=31)
    poison_unused_rows(case)
    out, kc, vc = gpu_chunk(case, mode)
    ref, kb, vb = oracle_chunk(case)
    # caches after the append are bit-identical (rows past each chunk untouched)
    assert np.array_equal(bf16_bits(kc), kb)
    assert np.array_equal(bf16_bits(vc), vb)
    check_bf16(out.float().cpu().numpy(), ref, f"chunk small ({mode})")


@pytest.mark.parametrize("heads,kv_heads", [(4, 4), (8, 1), (16, 2)])
def test_chunk_group_sizes(cuda_lib, heads, kv_heads):
    case = chunk_case(lengths=[200, 77, 256], pos=[300, 0, 128], cap=600, heads=heads, kv_heads=kv_heads,
                      seed=32)
    poison_unused_rows(case)
    out, _, _ = gpu_chunk(case)
    ref, _, _ = oracle_chunk(case)
    check_bf16(out.float().cpu().numpy(), ref, f"chunk H{heads}/{kv_heads}")


# (lengths, pos, cap, heads, kv_heads): tile edges in the chunk length and the
# offset, a chunk ending at the last cache row of a cap that is not a whole
# number of 128-key tiles (the widened rows are padded to whole tiles), one
# ending on a tile boundary (no zero rows after it), single-token chunks,
# position 0, GQA groups of 1, 3 and 8
BOTH_PATHS = [
    ([1, 5, 128, 129, 300, 0, 257, 64], [0, 200, 128, 126, 1000, 7, 383, 1536], 1600, 9, 3),
    ([100, 1, 1, 256], [900, 0, 999, 128], 1000, 8, 1),
    ([640, 3], [0, 637], 640, 4, 4),
]


@pytest.mark.parametrize("lengths,pos,cap,heads,kv_heads", BOTH_PATHS)
@pytest.mark.parametrize("mode", ["split", "step"])
def test_chunk_both_workspaces_match_the_oracle(cuda_lib, lengths, pos, cap, heads, kv_heads, mode):
    case = chunk_case(lengths=lengths, pos=pos, cap=cap, heads=heads, kv_heads=kv_heads, seed=37)
    poison_unused_rows(case)
    ref, kb, vb = oracle_chunk(case)
    for op in (2, 5):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, kc, vc = gpu_chunk(case, mode, dev_status=st, ws_op=op)
        assert int(st.item()) == 0, (op, int(st.item()))
        assert np.array_equal(bf16_bits(kc), kb) and np.array_equal(bf16_bits(vc), vb)
        check_bf16(out.float().cpu().numpy(), ref, f"chunk workspace op {op} ({mode})")


@pytest.mark.parametrize("ws_op,mode", [(2, "split"), (2, "step"), (5, "split"), (5, "step")])
def test_chunk_f16_range_flag(cuda_lib, ws_op, mode):
    # Both chunk paths round cached keys and values (the chunk's own rows
    # included, once appended) and the scaled rotated queries to f16 for the
    # tensor cores; beyond 65504 they saturate and KIME_DEV_RANGE is set.
    # Ordinary inputs leave it clear.
    case = chunk_case(lengths=[150, 40], pos=[300, 0], cap=512, seed=38)
    H, Hkv = case.heads, case.kv_heads
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _, _ = gpu_chunk(case, mode, dev_status=st, ws_op=ws_op)
    assert int(st.item()) == 0 and torch.isfinite(out.float()).all()
    for what in ("cached k", "cached v", "appended v", "q"):
        c2 = dataclasses.replace(case, qkv=case.qkv.clone(), k_cache=case.k_cache.clone(),
                                 v_cache=case.v_cache.clone())
        if what == "cached k":
            c2.k_cache[0, 1, 100, 5] = 1e5     # key 100 of sequence 0, below its pos
        elif what == "cached v":
            c2.v_cache[0, 0, 299, 7] = -1e5    # the last cached row before the chunk
        elif what == "appended v":
            c2.qkv[10, (H + Hkv) * 64 + 3] = 1e5   # chunk row 10 of sequence 0, value head 0
        else:
            c2.qkv[20, 3] = 5e5                # a query: 5e5 * 0.125 * log2(e) > 65504
        st.zero_()
        out, _, _ = gpu_chunk(c2, mode, dev_status=st, ws_op=ws_op)
        assert int(st.item()) == kime.DEV_RANGE, what
        assert torch.isfinite(out.float()).all(), what


def test_chunk_at_position_zero_matches_causal_prefill_oracle(cuda_lib):
    # pos = 0 everywhere: the chunk is a causal prefill whose keys went through
    # the cache (rounded to bf16 after rotation); against the chunk oracle it is
    # within the BF16 bound, and the two oracles agree to the rounding of k.
    case = chunk_case(lengths=[300, 129, 1], pos=[0, 0, 0], cap=512, seed=33)
    out, _, _ = gpu_chunk(case)
    ref, _, _ = oracle_chunk(case)
    check_bf16(out.float().cpu().numpy(), ref, "chunk pos 0")


def test_chunk_full_size_sampled(cuda_lib):
    case = chunk_case(device="cuda")
    out, kc, vc = gpu_chunk(case)
    assert torch.isfinite(out.float()).all()
    rows, heads = sample_items(case.cu_seqlens.numpy(), case.heads, 48, seed=6)
    cpu = dataclasses.replace(case, qkv=case.qkv.cpu(), k_cache=case.k_cache.cpu(), v_cache=case.v_cache.cpu())
    ref, kb, vb = oracle_chunk(cpu, rows=rows, heads=heads)
    got = out.float().cpu().numpy().reshape(case.total, case.heads, 64)[rows, heads]
    check_bf16(got, ref, "chunk full size")
    # every appended row (and every other cache row) is bit-identical to the oracle's
    assert np.array_equal(bf16_bits(kc), kb) and np.array_equal(bf16_bits(vc), vb)


def test_chunk_step_equals_append_then_attend_bitwise(cuda_lib):
    case = chunk_case(lengths=[333, 12, 700], pos=[17, 4000, 1024], cap=4096, seed=34)
    a, ka, va = gpu_chunk(case, "split")
    b, kb_, vb_ = gpu_chunk(case, "step")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ka.view(torch.int16), kb_.view(torch.int16))


def test_chunk_of_one_token_matches_decode(cuda_lib):
    # L = 1 chunks are decode steps: both paths against the same oracle values
    case = chunk_case(lengths=[1] * 6, pos=[0, 1, 127, 128, 999, 2047], cap=2048, seed=35)
    out, _, _ = gpu_chunk(case)
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.cap)
    kc, vc = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    dec = kime.kime_decode_step(case.qkv.to(dev), case.pos.to(dev), case.heads, case.kv_heads, kc, vc,
                                case.scale, c, s)
    ref, _, _ = oracle_chunk(case)
    check_bf16(out.float().cpu().numpy(), ref, "chunk L=1")
    check_bf16(dec.float().cpu().numpy(), ref, "decode step vs chunk oracle")


# ---- errors -------------------------------------------------------------------------

def test_chunk_bad_positions_are_reported_and_skipped(cuda_lib):
    case = chunk_case(lengths=[10, 20, 30], pos=[0, 90, 5], cap=100, seed=36)
    case.pos[1] = 81  # 81 + 20 > 100: refused before any write
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.cap)
    qkv, cu, pos = case.qkv.to(dev), case.cu_seqlens.to(dev), case.pos.to(dev)
    kc, vc = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full((case.total, case.heads * 64), 7.0, dtype=torch.bfloat16, device=dev)
    kime.kime_chunk_step(qkv, cu, pos, 30, case.heads, case.kv_heads, kc, vc, case.scale, c, s, out=out,
                         dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kime.DEV_BAD_POS
    assert torch.equal(kc[1].view(torch.int16), case.k_cache[1].to(dev).view(torch.int16))
    assert torch.equal(vc[1].view(torch.int16), case.v_cache[1].to(dev).view(torch.int16))
    assert bool((out[10:30].float() == 7.0).all())  # sequence 1's rows are not written
    # the other sequences are computed normally
    keep = [0, 2]
    rows = torch.cat([torch.arange(int(case.cu_seqlens[q]), int(case.cu_seqlens[q + 1])) for q in keep])
    sub = dataclasses.replace(case, lengths=[case.lengths[q] for q in keep],
                              cu_seqlens=torch.tensor([0, 10, 40], dtype=torch.int32), pos=case.pos[keep],
                              qkv=case.qkv[rows], k_cache=case.k_cache[keep], v_cache=case.v_cache[keep])
    ref, _, _ = oracle_chunk(sub)
    check_bf16(out[rows.to(dev)].float().cpu().numpy(), ref, "chunk beside a bad sequence")


def test_chunk_host_errors(cuda_lib):
    case = chunk_case(lengths=[8], pos=[0], cap=64, seed=37)
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.cap)
    qkv, cu, pos = case.qkv.to(dev), case.cu_seqlens.to(dev), case.pos.to(dev)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    with pytest.raises(kime.KimeError):  # heads not a multiple of kv_heads
        kime.kime_attn_chunk(qkv, cu, pos, 8, 9, 2, kc, vc, 0.125, c, s)
    with pytest.raises(kime.KimeError):  # scale must be positive
        kime.kime_attn_chunk(qkv, cu, pos, 8, 9, 3, kc, vc, 0.0, c, s)
    with pytest.raises(kime.KimeError):  # workspace too small
        kime.kime_attn_chunk(qkv, cu, pos, 8, 9, 3, kc, vc, 0.125, c, s,
                             workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    flat = torch.empty(qkv.numel() * 2 + 8, dtype=torch.uint8, device=dev)
    mis = flat[2:2 + qkv.numel() * 2].view(torch.bfloat16).view(qkv.shape)
    with pytest.raises(kime.KimeError):  # misaligned qkv
        kime.kime_kv_append_varlen(mis, cu, pos, 9, 3, kc, vc, c, s)


def test_chunk_of_empty_blocks_launches_nothing(cuda_lib):
    # every sequence has an empty block: no rows, nothing written, no error
    case = chunk_case(lengths=[0, 0, 0], pos=[5, 0, 63], cap=64, seed=38)
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, kc, vc = gpu_chunk(case, "step", dev_status=st)
    assert out.shape[0] == 0 and int(st.item()) == 0
    assert torch.equal(kc.view(torch.int16), case.k_cache.to(dev).view(torch.int16))
