"""Seeded synthetic inputs for the five workloads (and for small test shapes).

This module only draws random numbers into tensors of the right shapes; it
holds none of the attention arithmetic, so both the CUDA path and the oracle
can take their inputs from it.  Lengths are drawn first, then values, from a
``torch.Generator`` seeded per workload.

Workloads (head_dim 64 throughout):
  tiny              2 seqs (7, 13), 2 heads, FP32 qkv N(0,1), theta 1e4, full
  modernbert_base   64 seqs L~U[32,512], 12 heads, BF16 N(0,1.5^2);
                    local layer window 64 (128 wide) theta 1e4, global theta 1.6e5
  modernbert_large  8 seqs L~U[1024,8192], 16 heads, BF16 N(0,1.5^2); same layers
  smollm2_prefill   16 x 1142, 9 q / 3 kv heads, BF16 N(0,1), q part x 1/8,
                    theta 1e5, causal, scale 1
  smollm2_decode    128 seqs, 9 q / 3 kv heads, BF16 caches [128,3,8192,64]
                    N(0,1), used lengths pos~U[1,8191], theta 1e5, scale 1/8
  smollm2_chunk     chunked prefill: 32 seqs, 9 q / 3 kv heads, caches
                    [32,3,8192,64] N(0,1), chunks L~U[128,1024] of BF16 N(0,1)
                    rows at used lengths pos~U[0,8192-L], theta 1e5, scale 1/8
  smollm2_proj      the SmolLM2 prefill from the layer's input: 16 x 1142 token
                    rows x of hidden 576, BF16 N(0,1); one fused q/k/v weight
                    [960, 576] BF16 N(0, 1/576), its q rows x 1/8 (pre-scaled at
                    load); 9 q / 3 kv heads, theta 1e5, causal, scale 1
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass
class Layer:
    name: str
    window: int
    theta: float
    causal: bool
    scale: float


@dataclass
class VarlenCase:
    name: str
    lengths: list
    cu_seqlens: torch.Tensor  # int32 [n+1]
    qkv: torch.Tensor         # [T, 64*(H+2Hkv)]
    heads: int
    kv_heads: int
    layers: list = field(default_factory=list)

    @property
    def total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.lengths else 0


@dataclass
class DecodeCase:
    name: str
    pos: torch.Tensor       # int32 [n]
    qkv_new: torch.Tensor   # bf16 [n, W]
    k_cache: torch.Tensor   # bf16 [n, Hkv, cap, 64]
    v_cache: torch.Tensor
    heads: int
    kv_heads: int
    cap: int
    theta: float
    scale: float


@dataclass
class ChunkCase:
    name: str
    lengths: list
    cu_seqlens: torch.Tensor  # int32 [n+1]
    pos: torch.Tensor         # int32 [n]: cache rows already used
    qkv: torch.Tensor         # bf16 [T, W]: the chunks' rows
    k_cache: torch.Tensor     # bf16 [n, Hkv, cap, 64]
    v_cache: torch.Tensor
    heads: int
    kv_heads: int
    cap: int
    theta: float
    scale: float

    @property
    def total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.lengths else 0


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def random_qkv(lengths, heads, kv_heads, dtype, std, seed, device="cpu", q_scale=None):
    g = torch.Generator(device=device).manual_seed(seed)
    T = sum(int(x) for x in lengths)
    W = 64 * (heads + 2 * kv_heads)
    x = torch.randn((T, W), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x = x * std
    if q_scale is not None:
        x[:, : heads * 64] *= q_scale
    return x.to(dtype)


def _lengths(g, n, lo, hi):
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=g)]


def varlen_case(name: str, device: str = "cpu") -> VarlenCase:
    """One of the four prefill workloads; values are generated on `device`."""
    if name == "tiny":
        lengths, H, Hkv, dt, std, seed = [7, 13], 2, 2, torch.float32, 1.0, 1
        layers = [Layer("full", -1, 1e4, False, 0.125)]
        qs = None
    elif name == "modernbert_base":
        seed = 2
        lengths = _lengths(torch.Generator().manual_seed(seed), 64, 32, 512)
        H, Hkv, dt, std, qs = 12, 12, torch.bfloat16, 1.5, None
        layers = [Layer("local", 64, 1e4, False, 0.125), Layer("global", -1, 1.6e5, False, 0.125)]
    elif name == "modernbert_large":
        seed = 3
        lengths = _lengths(torch.Generator().manual_seed(seed), 8, 1024, 8192)
        H, Hkv, dt, std, qs = 16, 16, torch.bfloat16, 1.5, None
        layers = [Layer("local", 64, 1e4, False, 0.125), Layer("global", -1, 1.6e5, False, 0.125)]
    elif name == "smollm2_prefill":
        seed = 4
        lengths = [1142] * 16
        H, Hkv, dt, std, qs = 9, 3, torch.bfloat16, 1.0, 0.125
        layers = [Layer("causal", -1, 1e5, True, 1.0)]
    else:
        raise KeyError(name)
    qkv = random_qkv(lengths, H, Hkv, dt, std, seed * 1000 + 7, device=device, q_scale=qs)
    return VarlenCase(name, lengths, cu_from_lengths(lengths), qkv, H, Hkv, layers)


def decode_case(n_seqs: int = 128, cap: int = 8192, heads: int = 9, kv_heads: int = 3, seed: int = 5,
                device: str = "cpu", max_pos: int | None = None) -> DecodeCase:
    """The SmolLM2-shaped decode step (defaults) or a smaller one."""
    g = torch.Generator().manual_seed(seed)
    hi = cap - 1 if max_pos is None else max_pos
    pos = torch.randint(1, hi + 1, (n_seqs,), generator=g, dtype=torch.int64).to(torch.int32)
    gv = torch.Generator(device=device).manual_seed(seed * 1000 + 7)
    W = 64 * (heads + 2 * kv_heads)
    qkv_new = torch.randn((n_seqs, W), generator=gv, dtype=torch.float32, device=device).to(torch.bfloat16)
    k = torch.empty((n_seqs, kv_heads, cap, 64), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for s in range(n_seqs):  # per sequence, to bound the float32 temporaries
        k[s] = torch.randn((kv_heads, cap, 64), generator=gv, dtype=torch.float32, device=device)
        v[s] = torch.randn((kv_heads, cap, 64), generator=gv, dtype=torch.float32, device=device)
    return DecodeCase("smollm2_decode", pos, qkv_new, k, v, heads, kv_heads, cap, 1e5, 0.125)


@dataclass
class ProjCase:
    name: str
    lengths: list
    cu_seqlens: torch.Tensor  # int32 [n+1]
    x: torch.Tensor           # bf16 [T, hidden]
    w: torch.Tensor           # bf16 [64*(H+2Hkv), hidden]: q rows, k rows, v rows
    heads: int
    kv_heads: int
    theta: float
    window: int
    causal: bool
    scale: float

    @property
    def total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.lengths else 0


def random_proj(lengths, hidden, heads, kv_heads, seed, device="cpu", q_scale=None):
    """x [T, hidden] bf16 N(0,1) and a weight [64*(H+2Hkv), hidden] bf16
    N(0, 1/hidden) (projections of unit variance), q rows optionally scaled."""
    g = torch.Generator(device=device).manual_seed(seed)
    T = sum(int(v) for v in lengths)
    x = torch.randn((T, hidden), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
    w = torch.randn((64 * (heads + 2 * kv_heads), hidden), generator=g, dtype=torch.float32, device=device)
    w = w * (1.0 / hidden) ** 0.5
    if q_scale is not None:
        w[: heads * 64] *= q_scale
    return x, w.to(torch.bfloat16)


def proj_case(name: str = "smollm2_proj", device: str = "cpu") -> ProjCase:
    """The projection-fed SmolLM2 prefill workload."""
    if name != "smollm2_proj":
        raise KeyError(name)
    lengths = [1142] * 16
    x, w = random_proj(lengths, 576, 9, 3, 8 * 1000 + 7, device=device, q_scale=0.125)
    return ProjCase(name, lengths, cu_from_lengths(lengths), x, w, 9, 3, 1e5, -1, True, 1.0)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bfloat16 tensor (moved to the CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def chunk_case(n_seqs: int = 32, cap: int = 8192, lo: int = 128, hi: int = 1024, heads: int = 9,
               kv_heads: int = 3, seed: int = 6, device: str = "cpu", lengths=None, pos=None) -> ChunkCase:
    """The SmolLM2-shaped chunked-prefill step (defaults), a smaller one, or
    given lengths / positions.  Cache rows are N(0,1) everywhere (rows at and
    past pos are what the append overwrites or never reads)."""
    g = torch.Generator().manual_seed(seed)
    if lengths is None:
        lengths = _lengths(g, n_seqs, lo, hi)
    lengths = [int(x) for x in lengths]
    n = len(lengths)
    if pos is None:
        pos = [int(torch.randint(0, cap - L + 1, (1,), generator=g)) for L in lengths]
    pos = torch.tensor([int(x) for x in pos], dtype=torch.int32)
    gv = torch.Generator(device=device).manual_seed(seed * 1000 + 7)
    qkv = random_qkv(lengths, heads, kv_heads, torch.bfloat16, 1.0, seed * 1000 + 11, device=device)
    k = torch.empty((n, kv_heads, cap, 64), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for s in range(n):
        k[s] = torch.randn((kv_heads, cap, 64), generator=gv, dtype=torch.float32, device=device)
        v[s] = torch.randn((kv_heads, cap, 64), generator=gv, dtype=torch.float32, device=device)
    return ChunkCase("smollm2_chunk", lengths, cu_from_lengths(lengths), pos, qkv, k, v, heads, kv_heads, cap,
                     1e5, 0.125)
