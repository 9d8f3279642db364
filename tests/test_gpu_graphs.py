"""The entry points are CUDA-graph capturable: every launch goes on the given
stream, nothing is allocated or synchronised on the run path, and the
programmatic dependent launches (scheduler -> row preparation -> attention,
plan -> decode) become graph edges.  A captured call, replayed, gives the
bits of the direct call -- including after its inputs (positions, qkv rows)
are changed in place between replays."""
import pytest
import torch

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import chunk_case, cu_from_lengths, decode_case, random_qkv

from parity_util import gpu_tables

pytestmark = pytest.mark.gpu


def test_decode_step_replays_from_a_cuda_graph(cuda_lib):
    dev = torch.device("cuda")
    case = decode_case(n_seqs=16, cap=1024, seed=41)
    case.pos.copy_(torch.randint(0, 1000, (16,), generator=torch.Generator().manual_seed(41), dtype=torch.int32))
    n, H, Hkv, cap = len(case.pos), case.heads, case.kv_heads, case.cap
    c, s = gpu_tables(case.theta, cap)
    qn = case.qkv_new.to(dev)
    # direct: three steps, the positions advancing by one each
    kc1, vc1 = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    pos1 = case.pos.to(dev)
    want = []
    for _ in range(3):
        want.append(kime.kime_decode_step(qn, pos1, H, Hkv, kc1, vc1, case.scale, c, s).clone())
        pos1 += 1
    # captured once, replayed three times (first-call set-up done outside the capture)
    kc2, vc2 = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    pos2 = case.pos.to(dev)
    out = torch.empty((n, H * 64), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(kime.kime_attn_workspace_bytes(1, n, 0, H, Hkv, cap), dtype=torch.uint8, device=dev)
    kime.kime_decode_step(qn, pos2, H, Hkv, kc2.clone(), vc2.clone(), case.scale, c, s, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kime.kime_decode_step(qn, pos2, H, Hkv, kc2, vc2, case.scale, c, s, out=out, workspace=ws)
    for step in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want[step]), step
        pos2 += 1
    torch.cuda.synchronize()
    assert torch.equal(kc2, kc1) and torch.equal(vc2, vc1)


@pytest.mark.parametrize("op", [0, 3])
def test_varlen_replays_from_a_cuda_graph(cuda_lib, op):
    # op 0: the attention kernel does the RoPE; op 3: rows prepared first
    dev = torch.device("cuda")
    lengths, H, Hkv = [700, 1, 129, 300, 1500], 4, 2
    cu = cu_from_lengths(lengths).to(dev)
    T, n, mx = sum(lengths), len(lengths), max(lengths)
    c, s = gpu_tables(1e4, mx)
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=43).to(dev)
    ws = torch.empty(kime.kime_attn_workspace_bytes(op, n, T, H, Hkv), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H * 64), dtype=torch.bfloat16, device=dev)
    call = lambda o: kime.kime_attn_varlen(qkv, cu, mx, H, Hkv, -1, True, 0.125, c, s, out=o, workspace=ws)
    call(out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out)
    for seed in (44, 45):
        qkv.copy_(random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=seed).to(dev))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        want = call(torch.empty_like(out))
        torch.cuda.synchronize()
        assert torch.equal(out, want), seed


@pytest.mark.parametrize("op", [2, 5])  # the kernel that converts its own tiles; the one over prepared rows
def test_chunk_step_replays_from_a_cuda_graph(cuda_lib, op):
    dev = torch.device("cuda")
    case = chunk_case(n_seqs=6, cap=2048, lo=1, hi=300, seed=47)
    n, H, Hkv = len(case.lengths), case.heads, case.kv_heads
    c, s = gpu_tables(case.theta, case.cap)
    qkv, cu, pos = case.qkv.to(dev), case.cu_seqlens.to(dev), case.pos.to(dev)
    ws = torch.empty(kime.kime_attn_workspace_bytes(op, n, case.total, H, Hkv, case.cap), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((case.total, H * 64), dtype=torch.bfloat16, device=dev)
    step = lambda kc, vc, o: kime.kime_chunk_step(qkv, cu, pos, case.max_seqlen, H, Hkv, kc, vc, case.scale, c, s,
                                                 out=o, workspace=ws)
    kc1, vc1 = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    want = step(kc1, vc1, torch.empty_like(out)).clone()
    kc2, vc2 = case.k_cache.to(dev, copy=True), case.v_cache.to(dev, copy=True)
    step(kc2.clone(), vc2.clone(), out)  # first-call set-up, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(kc2, vc2, out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    assert torch.equal(kc2, kc1) and torch.equal(vc2, vc1)
