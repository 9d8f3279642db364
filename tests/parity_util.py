"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare with the tolerances the
contract states (FP32 path max abs 1e-5; BF16 path max abs 2e-2 and relative
L2 5e-3 against the FP64 oracle on the same BF16-valued inputs)."""
import numpy as np
import torch

import oracle
import packed_varlen_attention_kime_gb300 as kime
from packed_varlen_attention_kime_gb300.inputs import bf16_bits

F32_ATOL = 1e-5
BF16_ATOL = 2e-2
BF16_REL_L2 = 5e-3

_tables = {}


def gpu_tables(theta, length, device="cuda"):
    key = (float(theta), int(length), str(device))
    if key not in _tables:
        c, s = kime.kime_rope_tables(theta, length)
        _tables[key] = (c.to(device), s.to(device))
    return _tables[key]


def oracle_tables(theta, length):
    c, s = oracle.rope_tables_f32(theta, length)
    return c.astype(np.float64), s.astype(np.float64)


def oracle_input(qkv: torch.Tensor):
    if qkv.dtype == torch.bfloat16:
        return bf16_bits(qkv)
    return qkv.detach().cpu().numpy()


def run_gpu_varlen(qkv, cu, max_seqlen, H, Hkv, window, causal, scale, theta, rope_len=None,
                   dev_status=None):
    dev = torch.device("cuda")
    rope_len = rope_len or max(max_seqlen, 1)
    c, s = gpu_tables(theta, rope_len)
    out = kime.kime_attn_varlen(qkv.to(dev), cu.to(dev), max_seqlen, H, Hkv, window, causal, scale, c, s,
                                dev_status=dev_status)
    torch.cuda.synchronize()
    return out


def run_oracle_varlen(qkv, cu, H, Hkv, window, causal, scale, theta, rope_len, rows=None, heads=None):
    c, s = oracle_tables(theta, max(rope_len, 1))
    return oracle.attn_varlen(oracle_input(qkv), cu.numpy(), H, Hkv, window, causal, scale, c, s,
                              rows=rows, row_heads=heads)


def check_bf16(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= BF16_ATOL, f"{what}: max abs {err.max():.3e} > {BF16_ATOL}"
    assert rel <= BF16_REL_L2, f"{what}: rel L2 {rel:.3e} > {BF16_REL_L2}"
    return err.max(), rel


def check_f32(got, ref, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - np.asarray(ref, np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= F32_ATOL, f"{what}: max abs {err.max():.3e} > {F32_ATOL}"
    return err.max()


def sample_items(cu, heads, n_random, seed):
    """(rows, heads) to check at full size: the first and last row of every
    sequence and of every 128-row tile boundary neighbourhood, plus random rows."""
    rng = np.random.default_rng(seed)
    cu = np.asarray(cu)
    rows = []
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        rows += [a, b - 1]
        for t in range(a + 127, b, 128):
            rows += [t, min(t + 1, b - 1)]
    rows = np.array(rows, np.int64)
    if len(rows) > 4 * n_random:
        rows = rng.choice(rows, 4 * n_random, replace=False)
    rows = np.concatenate([rows, rng.integers(0, int(cu[-1]), n_random)])
    hs = rng.integers(0, heads, len(rows))
    return rows.astype(np.int32), hs.astype(np.int32)
