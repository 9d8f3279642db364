"""Masked keys on the GPU: a query's output never depends on the keys it does
not see (ffai-argus 0.7.3 src/text.rs, module doc: deleting the mask is
bit-identical to adding -inf), checked where it is not automatic -- masked keys
inside a key tile the query's tile visits (the causal diagonal tile, a
window's edge tiles); what a non-finite value in such a key's V row does; and
the f16 range flag of the BF16 path."""
import numpy as np
import pytest
import torch

import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import cu_from_lengths, random_qkv

from parity_util import gpu_tables

pytestmark = pytest.mark.gpu

OPS = (0, 3)  # the kernel that rotates in shared memory, the one over prepared rows


def _run(qkv, lengths, H, Hkv, window, causal, op, dev_status=None):
    dev = torch.device("cuda")
    cu = cu_from_lengths(lengths).to(dev)
    T, n, mx = qkv.shape[0], len(lengths), max(lengths)
    c, s = gpu_tables(1e4, mx)
    ws = torch.empty(kime.kime_attn_workspace_bytes(op, n, T, H, Hkv), dtype=torch.uint8, device=dev)
    out = kime.kime_attn_varlen(qkv.to(dev), cu, mx, H, Hkv, window, causal, 0.125, c, s, workspace=ws,
                                dev_status=dev_status)
    torch.cuda.synchronize()
    return out.cpu()


# (lengths, H, Hkv, window, causal, query rows, key rows masked for all of
# them and lying in a key tile those rows' query tile visits)
MASKED = [
    # causal: future keys of the diagonal tile (keys 128..255 for rows 128..255)
    ([300, 50], 3, 1, -1, True, (128, 160), (200, 256)),
    # window 64: rows 130..149 see keys 66..213; keys 215..255 lie in a
    # visited edge tile on either key-tile grid
    ([400, 70], 4, 2, 64, False, (130, 150), (215, 256)),
    # window 0: a row sees only itself; the rest of its tile is masked
    ([200, 33], 2, 2, 0, False, (10, 20), (30, 120)),
    # causal GQA with a window: both masks at once
    ([700, 20], 6, 2, 64, True, (300, 320), (321, 384)),
]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("lengths,H,Hkv,window,causal,qrows,krows", MASKED)
def test_masked_keys_in_visited_tiles_leave_outputs_bitwise(cuda_lib, op, lengths, H, Hkv, window, causal, qrows,
                                                            krows):
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=61)
    base = _run(qkv, lengths, H, Hkv, window, causal, op)
    # other finite keys and values for the masked rows (kv heads of every
    # group), large enough that a leak into the max or the sums would show
    g = torch.Generator().manual_seed(62)
    alt = qkv.clone()
    k0, k1 = krows
    kv = alt[k0:k1, H * 64:]
    alt[k0:k1, H * 64:] = (torch.randn(kv.shape, generator=g) * 40.0).to(torch.bfloat16)
    out = _run(alt, lengths, H, Hkv, window, causal, op)
    q0, q1 = qrows
    assert torch.equal(out[q0:q1], base[q0:q1])
    # (the perturbation is real: some row that sees those keys changed)
    assert not torch.equal(out, base)


@pytest.mark.parametrize("op", OPS)
def test_non_finite_masked_value_reaches_its_key_tile(cuda_lib, op):
    # Documented behaviour: the PV products take masked keys with probability
    # exactly 0, and 0 * NaN = NaN, so a NaN in the V row of a key that is
    # masked for a query still reaches that query's output when the query's
    # tile visits the key's tile.  Inputs must be finite.  Rows whose query
    # tile does not visit that key tile are untouched.
    lengths, H, Hkv = [300, 40], 2, 2
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=63)
    base = _run(qkv, lengths, H, Hkv, -1, True, op)
    bad = qkv.clone()
    bad[250, (H + Hkv) * 64:(H + Hkv) * 64 + 64] = float("nan")  # key 250's value, kv head 0
    out = _run(bad, lengths, H, Hkv, -1, True, op).float().reshape(-1, H, 64)
    ref = base.float().reshape(-1, H, 64)
    # query tile 0 (rows 0..127) never visits key tile 1: unchanged
    assert torch.equal(out[:128], ref[:128])
    # rows 128..249 of head 0: key 250 is masked (future) but in their
    # diagonal tile -- NaN
    assert torch.isnan(out[128:250, 0]).all()
    # head 1 reads kv head 1: unchanged; the other sequence: unchanged
    assert torch.equal(out[:, 1], ref[:, 1])
    assert torch.equal(out[300:], ref[300:])


@pytest.mark.parametrize("op", OPS)
def test_f16_range_flag(cuda_lib, op):
    # The BF16 path rounds rotated keys, scaled rotated queries and values to
    # f16 for the tensor cores; beyond 65504 they saturate and KIME_DEV_RANGE
    # is set.  Ordinary inputs leave it clear.
    dev = torch.device("cuda")
    lengths, H, Hkv = [150, 90], 2, 2
    qkv = random_qkv(lengths, H, Hkv, torch.bfloat16, 1.5, seed=64)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = _run(qkv, lengths, H, Hkv, -1, False, op, dev_status=st)
    assert int(st.item()) == 0 and torch.isfinite(out.float()).all()
    k_col, v_col = H * 64 + 5, (H + Hkv) * 64 + 7
    for col, val in ((k_col, 1e5), (v_col, -1e5), (3, 5e5)):  # a key, a value, a query (times 0.125 log2 e)
        big = qkv.clone()
        big[[7, 160], col] = val
        st.zero_()
        out = _run(big, lengths, H, Hkv, -1, False, op, dev_status=st)
        assert int(st.item()) == kime.DEV_RANGE, (col, val)
        assert torch.isfinite(out.float()).all()
    # a query of 1e5 stays in range once scaled by 0.125 log2(e): no flag
    small = qkv.clone()
    small[7, 3] = 1e5
    st.zero_()
    _run(small, lengths, H, Hkv, -1, False, op, dev_status=st)
    assert int(st.item()) == 0
