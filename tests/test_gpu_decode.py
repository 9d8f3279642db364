"""GPU parity of kime_kv_append and kime_attn_decode against the FP64 oracle,
through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import bf16_bits, decode_case

from parity_util import check_bf16, gpu_tables, oracle_tables

pytestmark = pytest.mark.gpu


def gpu_step(case, dev_status=None, fused=False):
    """Append then decode through the C ABI: two entry points, or the fused
    kime_decode_step."""
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.cap)
    qn, pos = case.qkv_new.to(dev), case.pos.to(dev)
    kc, vc = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    if fused:
        out = kime.kime_decode_step(qn, pos, case.heads, case.kv_heads, kc, vc, case.scale, c, s,
                                    dev_status=dev_status)
    else:
        kime.kime_kv_append(qn, pos, case.heads, case.kv_heads, kc, vc, c, s, dev_status=dev_status)
        out = kime.kime_attn_decode(qn, pos, case.heads, case.kv_heads, kc, vc, case.scale, c, s,
                                    dev_status=dev_status)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_step(case, seqs):
    """Oracle append + decode for the listed sequences only (their own caches)."""
    seqs = np.asarray(seqs)
    qn = bf16_bits(case.qkv_new)[seqs]
    pos = case.pos.numpy()[seqs]
    kb = bf16_bits(case.k_cache[torch.from_numpy(seqs).long()]).copy()
    vb = bf16_bits(case.v_cache[torch.from_numpy(seqs).long()]).copy()
    c32, s32 = oracle.rope_tables_f32(case.theta, case.cap)
    assert oracle.kv_append(qn, pos, case.heads, case.kv_heads, case.cap, c32, s32, kb, vb) == 0
    c, s = oracle_tables(case.theta, case.cap)
    out = oracle.attn_decode(qn, pos, case.heads, case.kv_heads, case.cap, case.scale, c, s, kb, vb)
    return out, kb, vb


@pytest.mark.parametrize("fused", [False, True])
def test_append_and_decode_small_all_outputs(cuda_lib, fused):
    case = decode_case(n_seqs=12, cap=700, seed=21)
    # empty history, 128-key chunk edges, the last row of the cache
    case.pos[:7] = torch.tensor([0, 1, 127, 128, 255, 256, 699], dtype=torch.int32)
    out, kc, vc = gpu_step(case, fused=fused)
    ref, kb, vb = oracle_step(case, np.arange(12))
    # the caches after append are bit-identical, canaries (every other row) untouched
    assert np.array_equal(bf16_bits(kc), kb)
    assert np.array_equal(bf16_bits(vc), vb)
    check_bf16(out.float().cpu().numpy(), ref, "decode small")


@pytest.mark.parametrize("heads,kv_heads", [(4, 4), (8, 1), (6, 3)])
def test_decode_group_sizes(cuda_lib, heads, kv_heads):
    case = decode_case(n_seqs=5, cap=1100, heads=heads, kv_heads=kv_heads, seed=22)
    out, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case, np.arange(5))
    check_bf16(out.float().cpu().numpy(), ref, f"decode H{heads}/{kv_heads}")


@pytest.mark.parametrize("fused", [False, True])
def test_decode_full_size_sampled(cuda_lib, fused):
    case = decode_case(device="cuda")
    out, kc, _ = gpu_step(case, fused=fused)
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(5)
    pos = case.pos.numpy()
    seqs = np.unique(np.concatenate([[int(np.argmax(pos)), int(np.argmin(pos))],
                                     rng.choice(len(pos), 10, replace=False)]))
    idx = torch.from_numpy(seqs).long().cuda()
    qn = bf16_bits(case.qkv_new)[seqs]
    kb = bf16_bits(case.k_cache[idx]).copy()
    vb = bf16_bits(case.v_cache[idx]).copy()
    p = pos[seqs].astype(np.int32)
    c32, s32 = oracle.rope_tables_f32(case.theta, case.cap)
    assert oracle.kv_append(qn, p, case.heads, case.kv_heads, case.cap, c32, s32, kb, vb) == 0
    c, s = oracle_tables(case.theta, case.cap)
    ref = oracle.attn_decode(qn, p, case.heads, case.kv_heads, case.cap, case.scale, c, s, kb, vb)
    check_bf16(out.float().cpu().numpy()[seqs], ref, "decode full")
    # the appended rows are bit-identical to the oracle's
    kcs = bf16_bits(kc[idx])
    for k in range(len(seqs)):
        assert np.array_equal(kcs[k][:, p[k]], kb[k][:, p[k]])


def test_bad_positions_are_flagged_and_skipped(cuda_lib):
    dev = torch.device("cuda")
    case = decode_case(n_seqs=4, cap=300, seed=23)
    case.pos[1] = 300   # == cap
    case.pos[2] = -5
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    k_before = case.k_cache.clone()
    out, kc, vc = gpu_step(case, dev_status=st, fused=True)
    assert int(st.item()) & kime.DEV_BAD_POS
    kc = kc.cpu()
    assert torch.equal(kc[1], k_before[1]) and torch.equal(kc[2], k_before[2])
    ref, _, _ = oracle_step(case, np.array([0, 3]))
    check_bf16(out.float().cpu().numpy()[[0, 3]], ref, "decode valid rows")


def test_decode_host_argument_errors(cuda_lib):
    dev = torch.device("cuda")
    case = decode_case(n_seqs=2, cap=64, heads=9, kv_heads=1, seed=24, max_pos=10)
    c, s = gpu_tables(case.theta, case.cap)
    with pytest.raises(kime.KimeError):  # heads/kv_heads = 9 > 8
        kime.kime_attn_decode(case.qkv_new.to(dev), case.pos.to(dev), 9, 1, case.k_cache.to(dev),
                              case.v_cache.to(dev), 0.125, c, s)


def test_decode_empty_batch_launches_nothing(cuda_lib):
    dev = torch.device("cuda")
    case = decode_case(n_seqs=1, cap=64, seed=25, max_pos=10)
    c, s = gpu_tables(case.theta, case.cap)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    empty_pos = torch.zeros(0, dtype=torch.int32, device=dev)
    out = kime.kime_decode_step(case.qkv_new.to(dev)[:0], empty_pos, case.heads, case.kv_heads, kc, vc,
                                case.scale, c, s)
    torch.cuda.synchronize()
    assert out.shape[0] == 0
    assert torch.equal(kc.view(torch.int16), case.k_cache.to(dev).view(torch.int16))
