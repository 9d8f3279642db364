"""GPU parity of the QKV projection (kime_qkv_proj) and of attention fed by
it with the projection fused into the attention producer
(kime_attn_varlen_proj), through the C ABI, against the FP64 oracle:
oracle.qkv_proj (x W^T, weight [out, in]) and oracle.attn_varlen_proj (that
projection in FP64, then the attention definition; nothing rounded between).

Tolerances: the projection's outputs are FP32 sums rounded to bf16, so
within half a bf16 ulp (at most 2^-8 relative: 8 significant bits) plus the
FP32 accumulation error of
`hidden` products; attention outputs meet the BF16 path's contract (max abs
2e-2, relative L2 5e-3)."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import bf16_bits, cu_from_lengths, proj_case, random_proj

from parity_util import check_bf16, gpu_tables, oracle_tables, sample_items

pytestmark = pytest.mark.gpu

PROJ_SHAPES = [
    # lengths, hidden, H, Hkv: ragged row tiles; 15, 6 and 5 heads (the last
    # column tile of 3 heads full, or holding 2)
    ([1, 127, 2], 576, 9, 3),
    ([128, 1, 300], 64, 2, 2),
    ([129, 255, 77], 192, 3, 1),
    ([1000], 768, 12, 12),
]


@pytest.mark.parametrize("lengths,hidden,H,Hkv", PROJ_SHAPES)
def test_qkv_proj_all_elements(cuda_lib, lengths, hidden, H, Hkv):
    x, w = random_proj(lengths, hidden, H, Hkv, seed=71)
    dev = torch.device("cuda")
    got = kime.kime_qkv_proj(x.to(dev), w.to(dev), H, Hkv)
    torch.cuda.synchronize()
    ref = oracle.qkv_proj(bf16_bits(x), bf16_bits(w))
    g = got.float().cpu().numpy().astype(np.float64)
    # FP32 accumulation of exact bf16 products: |error| <= hidden * u * sum |x w| with
    # u = 2^-23 (allowing the tensor core's FP32 adds to truncate), doubled for margin
    acc = np.abs(x.float().numpy().astype(np.float64)) @ np.abs(w.float().numpy().astype(np.float64)).T
    bound = 2.0 ** -8 * np.abs(ref) * (1 + 1e-6) + hidden * 2.0 ** -22 * acc
    assert np.all(np.abs(g - ref) <= bound + 1e-30)


PROJ_ATTN = [
    # lengths, hidden, H, Hkv, window, causal, scale, q weight scale
    ([300, 129, 5, 1], 576, 9, 3, -1, True, 1.0, 0.125),
    ([1, 2, 63, 64, 65, 127, 128, 129, 255], 128, 2, 2, -1, False, 0.125, None),
    ([400, 257], 192, 3, 1, 64, False, 0.125, None),
    ([700, 33], 64, 4, 2, 0, False, 0.125, None),
]


@pytest.mark.parametrize("lengths,hidden,H,Hkv,window,causal,scale,qs", PROJ_ATTN)
def test_attn_varlen_proj_all_elements(cuda_lib, lengths, hidden, H, Hkv, window, causal, scale, qs):
    x, w = random_proj(lengths, hidden, H, Hkv, seed=72, q_scale=qs)
    dev = torch.device("cuda")
    cu = cu_from_lengths(lengths)
    mx = max(lengths)
    c, s = gpu_tables(1e5, mx)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = kime.kime_attn_varlen_proj(x.to(dev), w.to(dev), cu.to(dev), mx, H, Hkv, window, causal, scale, c, s,
                                     dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    oc, os_ = oracle_tables(1e5, mx)
    ref = oracle.attn_varlen_proj(bf16_bits(x), bf16_bits(w), cu.numpy(), H, Hkv, window, causal, scale, oc, os_)
    check_bf16(got.float().cpu().numpy(), ref, f"proj+attn {lengths} w{window} c{causal}")


def test_attn_varlen_proj_smollm2_full_size_sampled(cuda_lib):
    case = proj_case()
    dev = torch.device("cuda")
    c, s = gpu_tables(case.theta, case.max_seqlen)
    got = kime.kime_attn_varlen_proj(case.x.to(dev), case.w.to(dev), case.cu_seqlens.to(dev), case.max_seqlen,
                                     case.heads, case.kv_heads, case.window, case.causal, case.scale, c, s)
    torch.cuda.synchronize()
    assert torch.isfinite(got.float()).all()
    rows, hs = sample_items(case.cu_seqlens.numpy(), case.heads, 300, seed=73)
    oc, os_ = oracle_tables(case.theta, case.max_seqlen)
    ref = oracle.attn_varlen_proj(bf16_bits(case.x), bf16_bits(case.w), case.cu_seqlens.numpy(), case.heads,
                                  case.kv_heads, case.window, case.causal, case.scale, oc, os_, rows=rows,
                                  row_heads=hs)
    g = got.float().cpu().reshape(case.total, case.heads, 64)[torch.from_numpy(rows).long(),
                                                             torch.from_numpy(hs).long()]
    check_bf16(g.numpy(), ref, "smollm2 proj+attn")


def test_fused_and_unfused_projection_agree_with_the_oracle(cuda_lib):
    # GEMM then attend (bf16 qkv written, then prepared and attended) against
    # the oracle on those bf16 qkv rows; the fused path against the oracle from x
    lengths, hidden, H, Hkv = [300, 129, 5], 576, 9, 3
    x, w = random_proj(lengths, hidden, H, Hkv, seed=74, q_scale=0.125)
    dev = torch.device("cuda")
    cu = cu_from_lengths(lengths)
    c, s = gpu_tables(1e5, 300)
    qkv = kime.kime_qkv_proj(x.to(dev), w.to(dev), H, Hkv)
    unfused = kime.kime_attn_varlen(qkv, cu.to(dev), 300, H, Hkv, -1, True, 1.0, c, s)
    fused = kime.kime_attn_varlen_proj(x.to(dev), w.to(dev), cu.to(dev), 300, H, Hkv, -1, True, 1.0, c, s)
    torch.cuda.synchronize()
    oc, os_ = oracle_tables(1e5, 300)
    ref_u = oracle.attn_varlen(bf16_bits(qkv), cu.numpy(), H, Hkv, -1, True, 1.0, oc, os_)
    ref_f = oracle.attn_varlen_proj(bf16_bits(x), bf16_bits(w), cu.numpy(), H, Hkv, -1, True, 1.0, oc, os_)
    check_bf16(unfused.float().cpu().numpy(), ref_u, "unfused")
    check_bf16(fused.float().cpu().numpy(), ref_f, "fused")


def test_projection_scale_fold_is_bitwise_on_gpu(cuda_lib):
    # argus Block::q: q weight pre-scaled by 1/8 with scale 1 equals the
    # unscaled weight with scale 1/8, bit for bit (power-of-two scaling
    # commutes with every rounding on the way)
    lengths, hidden, H, Hkv = [200, 57], 128, 6, 2
    x, w = random_proj(lengths, hidden, H, Hkv, seed=75)
    wf = w.clone()
    wf[: 64 * H] = (wf[: 64 * H].float() * 0.125).to(torch.bfloat16)
    dev = torch.device("cuda")
    cu = cu_from_lengths(lengths).to(dev)
    c, s = gpu_tables(1e5, 200)
    a = kime.kime_attn_varlen_proj(x.to(dev), w.to(dev), cu, 200, H, Hkv, -1, True, 0.125, c, s)
    b = kime.kime_attn_varlen_proj(x.to(dev), wf.to(dev), cu, 200, H, Hkv, -1, True, 1.0, c, s)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_projection_range_flag_and_argument_errors(cuda_lib):
    dev = torch.device("cuda")
    lengths, hidden, H, Hkv = [90, 40], 64, 2, 2
    x, w = random_proj(lengths, hidden, H, Hkv, seed=76)
    cu = cu_from_lengths(lengths).to(dev)
    c, s = gpu_tables(1e5, 90)
    xb = x.clone()
    xb[5, :] = 3.0e5  # projections far beyond the f16 range
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kime.kime_attn_varlen_proj(xb.to(dev), w.to(dev), cu, 90, H, Hkv, -1, False, 0.125, c, s, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kime.DEV_RANGE
    with pytest.raises(kime.KimeError):  # hidden not a multiple of 64
        kime.kime_qkv_proj(x[:, :48].contiguous().to(dev), w[:, :48].contiguous().to(dev), H, Hkv)
    with pytest.raises(kime.KimeError):  # workspace without room for the prepared rows
        kime.kime_attn_varlen_proj(x.to(dev), w.to(dev), cu, 90, H, Hkv, -1, False, 0.125, c, s,
                                   workspace=torch.empty(kime.kime_attn_workspace_bytes(0, 2, 130),
                                                         dtype=torch.uint8, device=dev))
