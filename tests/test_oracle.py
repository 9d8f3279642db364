"""Pins of the FP64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against an independent formulation (a dense numpy
brute force with an explicit -inf mask, complex-number rotation, torch's
bfloat16 rounding), a closed form, or an invariant stated on the source pages:

  ffai-argus 0.7.3 src/text.rs, module doc: skipping masked columns equals
      materialising -inf then softmax, bit for bit; the 1/8 scale fold is exact.
  ffai-argus tests: causal rows sum to one with an exactly-zero tail; a decode
      step (offset k_len-1) attends to the whole cache.
  ffai-argus TextTower::block: GQA fold = MHA with kv heads repeated.
  kime-cuda 0.0.3 src/plan.rs, fn rope_tables: the table recipe.
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
        got = otiles.classify(cu_of(case["lengths"]), case["causal"], case["window"])
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
