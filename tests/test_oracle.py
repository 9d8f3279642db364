"""Pins of the FP64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against an independent formulation (a dense numpy
brute force with an explicit -inf mask, complex-number rotation, torch's
bfloat16 rounding), a closed form, or an invariant stated on the source pages:

  ffai-argus 0.7.3 src/text.rs, module doc: skipping masked columns equals
      materialising -inf then softmax, bit for bit; the 1/8 scale fold is exact.
  ffai-argus tests: causal rows sum to one with an exactly-zero tail; a decode
      step (offset k_len-1) attends to the whole cache.
  ffai-argus TextTower::block: GQA fold = MHA with kv heads repeated; a block
      of new tokens at index_pos is appended to the cache, then attends it
      with CausalSoftmax offset index_pos.
  kime-cuda 0.0.3 src/plan.rs, fn rope_tables: the table recipe.
  ffai-argus Block::q and kime-cuda Op::Gemm: the QKV projection out = x W^T
      with one [out, in] weight, q rows then k then v; the q rows pre-scaled
      by 1/8, exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import tiles as otiles

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cu_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def make_qkv(lengths, H, Hkv, rng=RNG, std=1.0):
    T = int(sum(lengths))
    return rng.normal(0.0, std, size=(T, 64 * (H + 2 * Hkv)))


def tables64(theta, n):
    return oracle.rope_tables_f64(theta, n)


# ---- brute force (independent dense formulation) ------------------------------

def rotate_complex(x, c_rows, s_rows):
    """RoPE as complex multiplication z * (c + i s) with z_t = x_t + i x_{t+32}."""
    z = x[..., :32] + 1j * x[..., 32:]
    w = c_rows + 1j * s_rows
    zr = z * w
    return np.concatenate([zr.real, zr.imag], axis=-1)


def brute_attention(qkv, cu, H, Hkv, window, causal, scale, cos, sin):
    T = int(cu[-1])
    out = np.zeros((T, H * 64))
    G = H // Hkv
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        if L == 0:
            continue
        pos = np.arange(L)
        i = pos[:, None]
        j = pos[None, :]
        vis = np.ones((L, L), bool)
        if causal:
            vis &= j <= i
        if window >= 0:
            vis &= np.abs(i - j) <= window
        for h in range(H):
            g = h // G
            q = rotate_complex(qkv[a:b, h * 64:(h + 1) * 64], cos[:L], sin[:L])
            k = rotate_complex(qkv[a:b, (H + g) * 64:(H + g + 1) * 64], cos[:L], sin[:L])
            v = qkv[a:b, (H + Hkv + g) * 64:(H + Hkv + g + 1) * 64]
            S = scale * (q @ k.T)
            S = np.where(vis, S, -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            out[a:b, h * 64:(h + 1) * 64] = P @ v
    return out


# ---- RoPE ---------------------------------------------------------------------

def test_rope_matches_complex_rotation():
    c, s = tables64(10000.0, 50)
    for p in [0, 1, 7, 49]:
        x = RNG.normal(size=64)
        y = oracle.rope(x, c[p], s[p])
        np.testing.assert_allclose(y, rotate_complex(x, c[p], s[p]), rtol=0, atol=1e-14)


def test_rope_identity_at_position_zero():
    c, s = oracle.rope_tables_f32(10000.0, 4)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    x = RNG.normal(size=64)
    assert np.array_equal(oracle.rope(x, c[0].astype(np.float64), s[0].astype(np.float64)), x)


def test_rope_preserves_norm():
    c, s = tables64(160000.0, 9000)
    for p in [1, 100, 4097, 8191]:
        x = RNG.normal(size=64)
        y = oracle.rope(x, c[p], s[p])
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)


def test_rope_scores_depend_on_relative_position_only():
    c, s = tables64(10000.0, 5000)
    q, k = RNG.normal(size=64), RNG.normal(size=64)
    for p, pp, d in [(3, 10, 100), (500, 20, 4000), (0, 0, 4321)]:
        a = oracle.rope(q, c[p], s[p]) @ oracle.rope(k, c[pp], s[pp])
        b = oracle.rope(q, c[p + d], s[p + d]) @ oracle.rope(k, c[pp + d], s[pp + d])
        assert abs(a - b) < 1e-9


def test_rope_tables_f32_closed_forms():
    c, s = oracle.rope_tables_f32(10000.0, 8192)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    # column 0 has inverse frequency theta^0 = 1, so the angle is p exactly.
    p = np.arange(8192)
    assert np.array_equal(c[:, 0], np.cos(p.astype(np.float64)).astype(np.float32))
    assert np.array_equal(s[:, 0], np.sin(p.astype(np.float64)).astype(np.float32))


def test_rope_tables_f32_within_bound_of_exact():
    for theta in (1e4, 1e5, 1.6e5):
        c32, s32 = oracle.rope_tables_f32(theta, 8192)
        c64, s64 = oracle.rope_tables_f64(theta, 8192)
        p = np.arange(8192, dtype=np.float64)[:, None]
        inv = theta ** (-np.arange(32) * 2.0 / 64.0)
        # float32 inverse frequency (<= 1 ulp of the quotient and power) and the
        # float32 angle product (1/2 ulp of the angle): |d angle| bound.
        bound = p * inv * 4.0 * 2.0 ** -24 + np.spacing((p * inv).astype(np.float32)) / 2 + 2.0 ** -24
        assert np.all(np.abs(c32 - c64) <= bound + 1e-7)
        assert np.all(np.abs(s32 - s64) <= bound + 1e-7)


def test_bf16_rounding_matches_torch():
    x = np.concatenate([RNG.normal(size=2000).astype(np.float32) * 10,
                        # exact ties between two bfloat16 values (low half 0x8000)
                        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, 1.0, -3.5, 65504.0], np.float32)])
    ours = oracle.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---- attention -------------------------------------------------------------------

CASES = [
    # lengths, H, Hkv, window, causal
    ([5, 0, 8, 1], 2, 2, -1, False),
    ([6, 3], 3, 1, -1, True),
    ([8, 7], 3, 3, 2, False),
    ([8, 2, 5], 2, 1, 1, True),
    ([1, 1, 4], 3, 3, 0, False),
]


@pytest.mark.parametrize("lengths,H,Hkv,window,causal", CASES)
def test_oracle_matches_dense_brute_force(lengths, H, Hkv, window, causal):
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, Hkv)
    c, s = oracle.rope_tables_f32(10000.0, 16)
    c, s = c.astype(np.float64), s.astype(np.float64)
    got = oracle.attn_varlen(qkv, cu, H, Hkv, window, causal, 0.125, c, s)
    ref = brute_attention(qkv, cu, H, Hkv, window, causal, 0.125, c, s)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_oracle_bf16_and_f32_inputs_widen_exactly():
    lengths, H = [9, 4], 2
    cu = cu_of(lengths)
    x = torch.from_numpy(make_qkv(lengths, H, H)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    c, s = tables64(10000.0, 16)
    a = oracle.attn_varlen(bits, cu, H, H, -1, False, 0.125, c, s)
    b = oracle.attn_varlen(x.float().numpy(), cu, H, H, -1, False, 0.125, c, s)
    d = oracle.attn_varlen(x.double().numpy(), cu, H, H, -1, False, 0.125, c, s)
    assert np.array_equal(a, b) and np.array_equal(a, d)


@pytest.mark.parametrize("causal,window", [(True, -1), (False, 3), (True, 2), (False, -1)])
def test_mask_skip_is_bitwise_equal_to_minus_inf_softmax(causal, window):
    lengths, H = [13, 6], 2
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, H, std=1.5)
    c, s = tables64(10000.0, 16)
    skip = oracle.attn_varlen(qkv, cu, H, H, window, causal, 0.125, c, s, mode=0)
    full = oracle.attn_varlen(qkv, cu, H, H, window, causal, 0.125, c, s, mode=1)
    assert np.array_equal(skip, full)


def test_scale_fold_is_bitwise():
    lengths, H = [11, 5], 3
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, H)
    folded = qkv.copy()
    folded[:, : H * 64] *= 0.125
    c, s = tables64(10000.0, 16)
    a = oracle.attn_varlen(qkv, cu, H, H, -1, True, 0.125, c, s)
    b = oracle.attn_varlen(folded, cu, H, H, -1, True, 1.0, c, s)
    assert np.array_equal(a, b)


def test_window_at_least_length_equals_full_bitwise():
    lengths, H = [12, 3, 7], 2
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, H)
    c, s = tables64(10000.0, 16)
    full = oracle.attn_varlen(qkv, cu, H, H, -1, False, 0.125, c, s)
    for w in (11, 12, 1000):
        assert np.array_equal(oracle.attn_varlen(qkv, cu, H, H, w, False, 0.125, c, s), full)


def test_window_zero_and_single_key_return_v():
    lengths, H, Hkv = [1, 6, 1], 3, 1
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, Hkv)
    c, s = tables64(10000.0, 16)
    v = qkv[:, (H + Hkv) * 64:(H + Hkv + 1) * 64]
    w0 = oracle.attn_varlen(qkv, cu, H, Hkv, 0, False, 0.125, c, s)
    for h in range(H):
        assert np.array_equal(w0[:, h * 64:(h + 1) * 64], v)
    full = oracle.attn_varlen(qkv, cu, H, Hkv, -1, True, 0.125, c, s)
    for r in (0, 1, 7):  # L=1 sequences and the first row of a causal sequence
        for h in range(H):
            assert np.array_equal(full[r, h * 64:(h + 1) * 64], v[r])


def test_rows_sum_to_one_and_masked_tail_is_zero():
    lengths, H = [33], 2
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, H, std=1.5)
    c, s = tables64(10000.0, 40)
    for r in range(33):
        p = oracle.attn_probs(qkv, cu, H, H, -1, True, 0.125, c, s, r, 1)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p[r + 1:] == 0.0) and np.all(p[: r + 1] > 0.0)
    p = oracle.attn_probs(qkv, cu, H, H, 4, False, 0.125, c, s, 20, 0)
    assert np.all(p[:16] == 0.0) and np.all(p[25:] == 0.0) and np.all(p[16:25] > 0)


def test_gqa_equals_mha_with_repeated_kv_bitwise():
    lengths, H, Hkv = [10, 4], 6, 2
    G = H // Hkv
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, Hkv)
    q = qkv[:, : H * 64]
    k = qkv[:, H * 64:(H + Hkv) * 64].reshape(-1, Hkv, 64)
    v = qkv[:, (H + Hkv) * 64:].reshape(-1, Hkv, 64)
    kr = np.repeat(k, G, axis=1).reshape(-1, H * 64)
    vr = np.repeat(v, G, axis=1).reshape(-1, H * 64)
    mha = np.concatenate([q, kr, vr], axis=1)
    c, s = tables64(10000.0, 16)
    a = oracle.attn_varlen(qkv, cu, H, Hkv, -1, True, 0.125, c, s)
    b = oracle.attn_varlen(mha, cu, H, H, -1, True, 0.125, c, s)
    assert np.array_equal(a, b)


def test_sampled_rows_equal_full_computation():
    lengths, H, Hkv = [40, 17, 3], 4, 2
    cu = cu_of(lengths)
    qkv = make_qkv(lengths, H, Hkv)
    c, s = tables64(10000.0, 64)
    full = oracle.attn_varlen(qkv, cu, H, Hkv, 5, True, 0.125, c, s)
    rows = np.array([0, 39, 40, 56, 57, 59], np.int32)
    hs = np.array([0, 3, 1, 2, 3, 0], np.int32)
    part = oracle.attn_varlen(qkv, cu, H, Hkv, 5, True, 0.125, c, s, rows=rows, row_heads=hs)
    for k, (r, h) in enumerate(zip(rows, hs)):
        assert np.array_equal(part[k], full[r, h * 64:(h + 1) * 64])


# ---- KV append and decode ----------------------------------------------------

def bf16_round_np(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_kv_append_rotates_rounds_and_touches_only_the_row():
    n, H, Hkv, cap = 3, 6, 2, 20
    W = 64 * (H + 2 * Hkv)
    new = torch.randn(n, W, dtype=torch.float32).to(torch.bfloat16)
    bits = new.view(torch.int16).numpy().view(np.uint16)
    pos = np.array([0, 5, 19], np.int32)
    c, s = oracle.rope_tables_f32(1e5, 32)
    kc = RNG.integers(0, 65535, size=(n, Hkv, cap, 64), dtype=np.uint16)
    vc = RNG.integers(0, 65535, size=(n, Hkv, cap, 64), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.kv_append(bits, pos, H, Hkv, cap, c, s, kc, vc) == 0
    x = new.float().numpy()
    for si in range(n):
        P = pos[si]
        for g in range(Hkv):
            xk = x[si, (H + g) * 64:(H + g + 1) * 64]
            a, b = xk[:32], xk[32:]
            # numpy float32 arithmetic rounds after every operation
            y = np.concatenate([a * c[P] - b * s[P], b * c[P] + a * s[P]]).astype(np.float32)
            assert np.array_equal(kc[si, g, P], bf16_round_np(y))
            assert np.array_equal(vc[si, g, P], bits[si, (H + Hkv + g) * 64:(H + Hkv + g + 1) * 64])
    mask = np.ones(kc.shape, bool)
    for si in range(n):
        mask[si, :, pos[si]] = False
    assert np.array_equal(kc[mask], k0[mask]) and np.array_equal(vc[mask], v0[mask])
    # out-of-range positions write nothing
    bad = np.array([-1, cap, 3], np.int32)
    kc2, vc2 = kc.copy(), vc.copy()
    assert oracle.kv_append(bits, bad, H, Hkv, cap, c, s, kc2, vc2) == 2
    assert np.array_equal(kc2[:2], kc[:2]) and np.array_equal(vc2[:2], vc[:2])


def test_decode_matches_dense_brute_force():
    n, H, Hkv, cap = 4, 6, 2, 40
    G = H // Hkv
    W = 64 * (H + 2 * Hkv)
    new = torch.randn(n, W).to(torch.bfloat16)
    bits = new.view(torch.int16).numpy().view(np.uint16)
    kc = torch.randn(n, Hkv, cap, 64).to(torch.bfloat16)
    vc = torch.randn(n, Hkv, cap, 64).to(torch.bfloat16)
    kb = kc.view(torch.int16).numpy().view(np.uint16).copy()
    vb = vc.view(torch.int16).numpy().view(np.uint16).copy()
    pos = np.array([0, 1, 17, 39], np.int32)
    c32, s32 = oracle.rope_tables_f32(1e5, 64)
    oracle.kv_append(bits, pos, H, Hkv, cap, c32, s32, kb, vb)
    c, s = c32.astype(np.float64), s32.astype(np.float64)
    got = oracle.attn_decode(bits, pos, H, Hkv, cap, 0.125, c, s, kb, vb)
    kf = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).double().numpy()
    vf = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).double().numpy()
    x = new.double().numpy()
    for si in range(n):
        P = pos[si]
        for h in range(H):
            g = h // G
            q = rotate_complex(x[si, h * 64:(h + 1) * 64], c[P], s[P])
            sc = 0.125 * (kf[si, g, : P + 1] @ q)
            p = np.exp(sc - sc.max())
            assert np.all(p > 0)  # the whole cache is attended
            ref = (p / p.sum()) @ vf[si, g, : P + 1]
            np.testing.assert_allclose(got[si, h * 64:(h + 1) * 64], ref, rtol=0, atol=1e-12)


def test_decode_equals_last_row_of_causal_prefill_bitwise():
    # With identity tables (cos 1, sin 0) the cached keys equal the raw keys, so
    # decode at position P is the last row of causal prefill over P+1 tokens.
    H, Hkv, P = 6, 2, 23
    L = P + 1
    W = 64 * (H + 2 * Hkv)
    x = torch.randn(L, W).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    ones = np.ones((L, 32), np.float32)
    zeros = np.zeros((L, 32), np.float32)
    cap = L + 3
    kb = np.zeros((1, Hkv, cap, 64), np.uint16)
    vb = np.zeros((1, Hkv, cap, 64), np.uint16)
    for g in range(Hkv):
        kb[0, g, :P] = bits[:P, (H + g) * 64:(H + g + 1) * 64]
        vb[0, g, :P] = bits[:P, (H + Hkv + g) * 64:(H + Hkv + g + 1) * 64]
    oracle.kv_append(bits[P:P + 1], np.array([P], np.int32), H, Hkv, cap, ones, zeros, kb, vb)
    dec = oracle.attn_decode(bits[P:P + 1], np.array([P], np.int32), H, Hkv, cap, 0.125,
                             ones.astype(np.float64), zeros.astype(np.float64), kb, vb)
    pre = oracle.attn_varlen(bits, np.array([0, L], np.int32), H, Hkv, -1, True, 0.125,
                             ones.astype(np.float64), zeros.astype(np.float64))
    assert np.array_equal(dec[0], pre[P])


# ---- tile classification ----------------------------------------------------------

def test_tile_classification_golden():
    with open(os.path.join(GOLDEN, "tiles_small.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        got = otiles.classify(cu_of(case["lengths"]), case["causal"], case["window"], pos=case.get("pos"))
        want = {(int(k.split(",")[0]), int(k.split(",")[1])): v for k, v in case["codes"].items()}
        assert set(got) == set(want), case["name"]
        for key, codes in want.items():
            assert got[key].tolist() == codes, (case["name"], key)


def test_tile_classification_is_two_nested_intervals():
    # The scheduler stores visited and full tiles as ranges; the brute-force
    # classification must have that shape for every mode.
    lengths = [1, 127, 128, 129, 255, 256, 300, 700]
    for causal in (False, True):
        for window in (-1, 0, 1, 63, 64, 65, 127, 128, 200, 1000):
            for (s, qt), codes in otiles.classify(cu_of(lengths), causal, window).items():
                vis = np.flatnonzero(codes > 0)
                full = np.flatnonzero(codes == 2)
                assert len(vis) > 0 and np.all(np.diff(vis) == 1)
                if len(full):
                    assert np.all(np.diff(full) == 1)
    for pos in ([0] * 8, [5, 0, 127, 128, 129, 1000, 3, 255]):
        for (s, qt), codes in otiles.classify(cu_of(lengths), True, -1, pos=pos).items():
            vis = np.flatnonzero(codes > 0)
            full = np.flatnonzero(codes == 2)
            assert len(vis) > 0 and np.all(np.diff(vis) == 1)
            if len(full):
                assert np.all(np.diff(full) == 1)


# ---- chunked prefill against the cache ------------------------------------------

def bf16_from_bits(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def chunk_setup(lengths, pos, H, Hkv, cap, theta=1e5, seed=0):
    """Random bf16 chunk rows, caches holding random already-rotated keys and
    values below each sequence's pos (garbage above), float32 tables."""
    g = torch.Generator().manual_seed(seed)
    T = int(sum(lengths))
    x = torch.randn(T, 64 * (H + 2 * Hkv), generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    n = len(lengths)
    kb = torch.randn(n, Hkv, cap, 64, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    vb = torch.randn(n, Hkv, cap, 64, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    c32, s32 = oracle.rope_tables_f32(theta, cap)
    return bits, kb, vb, c32, s32


def test_kv_append_varlen_rotates_rounds_and_touches_only_its_rows():
    lengths, pos = [3, 0, 5, 1], np.array([0, 7, 10, 19], np.int32)
    H, Hkv, cap = 6, 2, 20
    bits, kb, vb, c, s = chunk_setup(lengths, pos, H, Hkv, cap)
    k0, v0 = kb.copy(), vb.copy()
    cu = cu_of(lengths)
    assert oracle.kv_append_varlen(bits, cu, pos, H, Hkv, cap, c, s, kb, vb) == 0
    x = bf16_from_bits(bits).astype(np.float32)
    touched = np.zeros(kb.shape, bool)
    for si, L in enumerate(lengths):
        for i in range(L):
            r, P = cu[si] + i, pos[si] + i
            for g in range(Hkv):
                xk = x[r, (H + g) * 64:(H + g + 1) * 64]
                a, b = xk[:32], xk[32:]
                y = np.concatenate([a * c[P] - b * s[P], b * c[P] + a * s[P]]).astype(np.float32)
                assert np.array_equal(kb[si, g, P], bf16_round_np(y))
                assert np.array_equal(vb[si, g, P], bits[r, (H + Hkv + g) * 64:(H + Hkv + g + 1) * 64])
            touched[si, :, P] = True
    assert np.array_equal(kb[~touched], k0[~touched]) and np.array_equal(vb[~touched], v0[~touched])
    # a sequence whose block would leave [0, cap) (or the tables) writes nothing
    kb2, vb2 = k0.copy(), v0.copy()
    bad = np.array([-1, 7, 16, 19], np.int32)  # seq 0 negative, seq 2: 16 + 5 > 20
    assert oracle.kv_append_varlen(bits, cu, bad, H, Hkv, cap, c, s, kb2, vb2) == 2
    assert np.array_equal(kb2[[0, 2]], k0[[0, 2]]) and np.array_equal(vb2[[0, 2]], v0[[0, 2]])
    assert not np.array_equal(kb2[3], k0[3])
    short_c, short_s = c[:20], s[:20]
    kb3, vb3 = k0.copy(), v0.copy()
    assert oracle.kv_append_varlen(bits, cu, pos, H, Hkv, cap, short_c[:19], short_s[:19], kb3, vb3) == 1


def test_chunk_matches_dense_brute_force():
    lengths, pos = [4, 1, 0, 7], np.array([0, 9, 3, 25], np.int32)
    H, Hkv, cap = 6, 2, 40
    G = H // Hkv
    bits, kb, vb, c32, s32 = chunk_setup(lengths, pos, H, Hkv, cap, seed=3)
    cu = cu_of(lengths)
    oracle.kv_append_varlen(bits, cu, pos, H, Hkv, cap, c32, s32, kb, vb)
    c, s = c32.astype(np.float64), s32.astype(np.float64)
    got = oracle.attn_chunk(bits, cu, pos, H, Hkv, cap, 0.125, c, s, kb, vb)
    kf, vf, x = bf16_from_bits(kb), bf16_from_bits(vb), bf16_from_bits(bits)
    for si, L in enumerate(lengths):
        if L == 0:
            continue
        P = pos[si] + np.arange(L)
        Lk = pos[si] + L
        vis = np.arange(Lk)[None, :] <= P[:, None]
        for h in range(H):
            g = h // G
            q = rotate_complex(x[cu[si]:cu[si + 1], h * 64:(h + 1) * 64], c[P], s[P])
            S = np.where(vis, 0.125 * (q @ kf[si, g, :Lk].T), -np.inf)
            Pm = np.exp(S - S.max(axis=1, keepdims=True))
            ref = (Pm / Pm.sum(axis=1, keepdims=True)) @ vf[si, g, :Lk]
            np.testing.assert_allclose(got[cu[si]:cu[si + 1], h * 64:(h + 1) * 64], ref, rtol=0, atol=1e-12)


def test_chunk_equals_trailing_rows_of_causal_prefill_bitwise():
    # Identity tables (cos 1, sin 0): a cache holding the raw keys of tokens
    # 0..pos-1 plus a chunk of the next L tokens is causal prefill over pos+L
    # tokens, whose last L rows the chunk must reproduce bit for bit.
    H, Hkv = 6, 2
    seqs = [(0, 5), (17, 1), (40, 9)]  # (pos, L)
    cap = 64
    g = torch.Generator().manual_seed(11)
    W = 64 * (H + 2 * Hkv)
    full = [torch.randn(p + L, W, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            for p, L in seqs]
    ones, zeros = np.ones((cap, 32), np.float32), np.zeros((cap, 32), np.float32)
    kb = np.zeros((len(seqs), Hkv, cap, 64), np.uint16)
    vb = np.zeros((len(seqs), Hkv, cap, 64), np.uint16)
    for si, (p, L) in enumerate(seqs):
        for gg in range(Hkv):
            kb[si, gg, :p] = full[si][:p, (H + gg) * 64:(H + gg + 1) * 64]
            vb[si, gg, :p] = full[si][:p, (H + Hkv + gg) * 64:(H + Hkv + gg + 1) * 64]
    chunk = np.concatenate([f[p:] for f, (p, L) in zip(full, seqs)])
    cu = cu_of([L for p, L in seqs])
    pos = np.array([p for p, L in seqs], np.int32)
    assert oracle.kv_append_varlen(chunk, cu, pos, H, Hkv, cap, ones, zeros, kb, vb) == 0
    got = oracle.attn_chunk(chunk, cu, pos, H, Hkv, cap, 0.125, ones.astype(np.float64),
                            zeros.astype(np.float64), kb, vb)
    for si, (p, L) in enumerate(seqs):
        pre = oracle.attn_varlen(full[si], np.array([0, p + L], np.int32), H, Hkv, -1, True, 0.125,
                                 ones.astype(np.float64), zeros.astype(np.float64))
        assert np.array_equal(got[cu[si]:cu[si + 1]], pre[p:])


def test_chunk_split_in_two_is_bitwise_equal():
    # Prefilling a block in one chunk or in two consecutive chunks (the second
    # at pos + L1) leaves the same cache and gives the same rows, bit for bit.
    lengths, pos = [9, 6], np.array([3, 0], np.int32)
    H, Hkv, cap = 4, 2, 32
    bits, kb, vb, c32, s32 = chunk_setup(lengths, pos, H, Hkv, cap, seed=5)
    c, s = c32.astype(np.float64), s32.astype(np.float64)
    cu = cu_of(lengths)
    k1, v1 = kb.copy(), vb.copy()
    oracle.kv_append_varlen(bits, cu, pos, H, Hkv, cap, c32, s32, k1, v1)
    one = oracle.attn_chunk(bits, cu, pos, H, Hkv, cap, 0.125, c, s, k1, v1)
    split = [4, 2]
    first = np.concatenate([bits[cu[i]:cu[i] + split[i]] for i in range(2)])
    second = np.concatenate([bits[cu[i] + split[i]:cu[i + 1]] for i in range(2)])
    cu1, cu2 = cu_of(split), cu_of([lengths[i] - split[i] for i in range(2)])
    pos2 = pos + np.array(split, np.int32)
    k2, v2 = kb.copy(), vb.copy()
    oracle.kv_append_varlen(first, cu1, pos, H, Hkv, cap, c32, s32, k2, v2)
    a = oracle.attn_chunk(first, cu1, pos, H, Hkv, cap, 0.125, c, s, k2, v2)
    oracle.kv_append_varlen(second, cu2, pos2, H, Hkv, cap, c32, s32, k2, v2)
    b = oracle.attn_chunk(second, cu2, pos2, H, Hkv, cap, 0.125, c, s, k2, v2)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    for i in range(2):
        assert np.array_equal(one[cu[i]:cu[i] + split[i]], a[cu1[i]:cu1[i + 1]])
        assert np.array_equal(one[cu[i] + split[i]:cu[i + 1]], b[cu2[i]:cu2[i + 1]])


def test_chunk_of_one_token_equals_decode_bitwise():
    lengths, pos = [1, 1, 1], np.array([0, 13, 30], np.int32)
    H, Hkv, cap = 6, 3, 31
    bits, kb, vb, c32, s32 = chunk_setup(lengths, pos, H, Hkv, cap, seed=8)
    c, s = c32.astype(np.float64), s32.astype(np.float64)
    k1, v1, k2, v2 = kb.copy(), vb.copy(), kb.copy(), vb.copy()
    oracle.kv_append_varlen(bits, cu_of(lengths), pos, H, Hkv, cap, c32, s32, k1, v1)
    oracle.kv_append(bits, pos, H, Hkv, cap, c32, s32, k2, v2)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    ch = oracle.attn_chunk(bits, cu_of(lengths), pos, H, Hkv, cap, 0.125, c, s, k1, v1)
    dec = oracle.attn_decode(bits, pos, H, Hkv, cap, 0.125, c, s, k2, v2)
    assert np.array_equal(ch, dec)


def test_chunk_sampled_rows_equal_full_computation():
    lengths, pos = [5, 3], np.array([2, 11], np.int32)
    H, Hkv, cap = 4, 1, 16
    bits, kb, vb, c32, s32 = chunk_setup(lengths, pos, H, Hkv, cap, seed=9)
    c, s = c32.astype(np.float64), s32.astype(np.float64)
    cu = cu_of(lengths)
    oracle.kv_append_varlen(bits, cu, pos, H, Hkv, cap, c32, s32, kb, vb)
    full = oracle.attn_chunk(bits, cu, pos, H, Hkv, cap, 0.125, c, s, kb, vb)
    rows, heads = np.array([0, 4, 5, 7], np.int32), np.array([3, 0, 2, 1], np.int32)
    part = oracle.attn_chunk(bits, cu, pos, H, Hkv, cap, 0.125, c, s, kb, vb, rows=rows, row_heads=heads)
    for k, (r, h) in enumerate(zip(rows, heads)):
        assert np.array_equal(part[k], full[r, h * 64:(h + 1) * 64])
    with pytest.raises(ValueError):
        oracle.attn_chunk(bits, cu, np.array([2, 14], np.int32), H, Hkv, cap, 0.125, c, s, kb, vb)


# ---- QKV projection (the step before attention) ----------------------------------

def bf16_of(a):
    """float array -> bfloat16 bits (values chosen exactly representable, or rounded)."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def widen(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)


def test_qkv_proj_golden():
    # hand-derived: out[t][o] = sum_k x[t][k] w[o][k] with w stored [out, in]
    with open(os.path.join(GOLDEN, "qkv_proj_small.json")) as f:
        g = json.load(f)
    got = oracle.qkv_proj(bf16_of(g["x"]), bf16_of(g["w"]))
    assert np.array_equal(got, np.array(g["out"]))


def test_qkv_proj_selection_weights_pick_columns_exactly():
    # w[o] = unit row e_{perm[o]}: output column o is input column perm[o],
    # exactly -- a transposed weight or a swapped index would pick others
    rng = np.random.default_rng(7)
    x = bf16_of(rng.normal(size=(37, 128)))
    perm = rng.permutation(128)[:96]
    w = np.zeros((96, 128), np.float32)
    w[np.arange(96), perm] = 1.0
    got = oracle.qkv_proj(x, bf16_of(w))
    assert np.array_equal(got, widen(x)[:, perm])


def test_qkv_proj_matches_dense_numpy():
    # an independent formulation: numpy's dense product of the widened operands
    rng = np.random.default_rng(8)
    x = bf16_of(rng.normal(size=(53, 192)))
    w = bf16_of(rng.normal(scale=0.07, size=(320, 192)))
    ref = widen(x) @ widen(w).T
    got = oracle.qkv_proj(x, w)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert oracle.qkv_proj(x[:0], w).shape == (0, 320)


def test_projection_scale_fold_is_bitwise():
    # argus Block::q: the q weight pre-scaled by 1/8 at load, with scale 1,
    # equals the unscaled weight with scale 1/8 bit for bit (a power of two)
    rng = np.random.default_rng(9)
    lengths, H, Hkv, hidden = [19, 7, 33], 3, 1, 64
    T = sum(lengths)
    x = bf16_of(rng.normal(size=(T, hidden)))
    wf = rng.normal(scale=0.125, size=(64 * (H + 2 * Hkv), hidden)).astype(np.float32)
    w = bf16_of(wf)
    w_fold = widen(w).astype(np.float32)
    w_fold[: 64 * H] *= 0.125
    w_fold = bf16_of(w_fold)
    c, s = tables64(1e5, 64)
    a = oracle.attn_varlen_proj(x, w, cu_of(lengths), H, Hkv, -1, True, 0.125, c, s)
    b = oracle.attn_varlen_proj(x, w_fold, cu_of(lengths), H, Hkv, -1, True, 1.0, c, s)
    assert np.array_equal(a, b)


def test_projection_gqa_blocks():
    # the weight's rows are q heads, then k heads, then v heads: zeroing the
    # v rows of kv head 1 zeroes exactly the outputs of the q heads of group 1
    rng = np.random.default_rng(10)
    lengths, H, Hkv, hidden = [12, 9], 4, 2, 64
    T = sum(lengths)
    x = bf16_of(rng.normal(size=(T, hidden)))
    w = widen(bf16_of(rng.normal(scale=0.125, size=(64 * (H + 2 * Hkv), hidden)))).astype(np.float32)
    c, s = tables64(1e4, 16)
    base = oracle.attn_varlen_proj(x, bf16_of(w), cu_of(lengths), H, Hkv, -1, False, 0.125, c, s)
    w2 = w.copy()
    v1 = 64 * (H + Hkv + 1)
    w2[v1:v1 + 64] = 0.0
    out = oracle.attn_varlen_proj(x, bf16_of(w2), cu_of(lengths), H, Hkv, -1, False, 0.125, c, s)
    G = H // Hkv
    for h in range(H):
        blk = slice(h * 64, (h + 1) * 64)
        if h // G == 1:
            assert np.all(out[:, blk] == 0.0)
        else:
            assert np.array_equal(out[:, blk], base[:, blk])
