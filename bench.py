"""Benchmark of the packed-varlen attention hot path on GB300.

One step = the attention of one ModernBERT-large-shaped encoder layer pair
over one packed batch (8 sequences, lengths U[1024,8192], ~38.7k tokens, 16
heads x 64, BF16 qkv N(0, 1.5^2)): the local layer (window 64, RoPE theta
1e4) then the global layer (full, theta 1.6e5), each one kime_attn_varlen
call (device scheduler, row preparation, tcgen05 attention kernel).  Inputs
are resident in HBM before the timed region and L2 is flushed before every
timed step (a 512 MB write, then a 256 MB read that leaves only clean lines in
L2).

The same run also times, outside the headline number, each as the median of
200 flushed repetitions after 20 warm-ups: ModernBERT-base-shaped layers (64 x
U[32,512], the HBM-bound workload), SmolLM2-shaped causal GQA prefill (16 x
1142), the same prefill fed by its QKV projection (fused into the attention
producer, and projection-then-attend), the SmolLM2-shaped decode step (KV
append + split-KV decode, 128 sequences, cache 8192), chunked prefill, and
the FP32-qkv paths -- the "extra" object -- and the FP64 CPU oracle on a
bounded sample of the headline workload (cpu_baseline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extra]

Under torchrun every rank runs the same workload on its own GPU with no
exchange between ranks (weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("packed-varlen attention tokens/s & TFLOP/s (% BF16 peak); decode GB/s (% HBM) at 1 GB300")
HEADLINE = "modernbert_large"  # the largest single-GPU configuration: 8 x U[1024,8192] tokens, 16 heads
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one kime_attn_varlen call -- the sum over its
# kernels (scheduler, row preparation, attention kernel over prepared rows),
# from one ncu capture of each workload's layer (profiles/), keyed by the
# SHA-1 of those kernels' sources and the header they share: any change to
# them makes the figure stale, and the bench then reports null.
MEASURED_TRAFFIC = {
    ("6712770adf67b0b305683378dc5a761daab7ea70", "modernbert_large:global"): 769132032,
    ("6712770adf67b0b305683378dc5a761daab7ea70", "modernbert_base:global"): 240812544,
}
TRAFFIC_SOURCES = ("kime_common.cuh", "schedule.cu", "prep.cu", "prefill_rows.cu")


def traffic_key():
    import hashlib
    h = hashlib.sha1()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "packed_varlen_attention_kime_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload):
    return MEASURED_TRAFFIC.get((traffic_key(), workload))


# ---- helpers ---------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        out = {}
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            if v is not None:
                out[k] = float(v)
        if "hbm_gbs" in out and "bf16_tflops" in out:
            return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def visible_pairs(lengths, window, causal):
    """Exact number of (query, key) pairs attended, summed over sequences."""
    tot = 0
    for L in lengths:
        i = np.arange(L)
        if window < 0:
            hi = i if causal else np.full(L, L - 1)
            lo = np.zeros(L, np.int64)
        else:
            hi = np.minimum(i if causal else i + window, L - 1)
            lo = np.maximum(i - window, 0)
        tot += int((hi - lo + 1).sum())
    return tot


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(getattr(self, "text", ""))) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over the ranks of the default process group (the
    value itself when there is none): the job's time is its slowest rank's."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def l2_flush_buffer(dev):
    return torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)


def flush_l2(flush):
    """Evicts the step's data from the 129 MB L2: a 512 MB write, then a read of
    the buffer's first 256 MB (long evicted by the write), so the lines left
    in L2 are clean -- the write's last 129 MB would otherwise be written back
    to HBM inside the timed step."""
    flush.zero_()
    flush[: 256 * 1024 * 1024].max()


# ---- workloads on the GPU ------------------------------------------------------------

_STATUS = {}


def dev_status(dev):
    """The device status word every library call of this process reports into."""
    key = str(dev)
    if key not in _STATUS:
        _STATUS[key] = torch.zeros(1, dtype=torch.int32, device=dev)
    return _STATUS[key]


def check_status(dev):
    """Fails the run if any kernel flagged bad input or a timed-out wait."""
    torch.cuda.synchronize(dev)
    v = int(dev_status(dev).item())
    if v != 0:
        raise RuntimeError(f"device status {v:#x} after the timed work (a kernel flagged an error)")


class VarlenRun:
    """Device-resident inputs, tables, outputs and workspace for one varlen workload."""

    def __init__(self, name, dev, seed_offset=0):
        import packed_varlen_attention_kime_gb300 as kime
        from packed_varlen_attention_kime_gb300.inputs import varlen_case
        self.kime = kime
        self.case = varlen_case(name, device=str(dev))
        c = self.case
        self.dev = dev
        self.cu = c.cu_seqlens.to(dev)
        self.tables = {}
        for lay in c.layers:
            if lay.theta not in self.tables:
                cs, sn = kime.kime_rope_tables(lay.theta, c.max_seqlen)
                self.tables[lay.theta] = (cs.to(dev), sn.to(dev))
        self.outs = [torch.empty((c.total, c.heads * 64), dtype=c.qkv.dtype, device=dev) for _ in c.layers]
        # the workspace that lets the library prepare the qkv rows once per call (op 3)
        self.ws = torch.empty(kime.kime_attn_workspace_bytes(3, len(c.lengths), c.total, c.heads, c.kv_heads),
                              dtype=torch.uint8,
                              device=dev)
        self.flops = [4 * 64 * c.heads * visible_pairs(c.lengths, l.window, l.causal) for l in c.layers]
        W = c.qkv.shape[1]
        self.bytes_per_layer = c.total * W * 2 + c.total * c.heads * 64 * 2  # qkv read + out written

    def layer(self, k, qkv=None, out=None):
        c, lay = self.case, self.case.layers[k]
        cs, sn = self.tables[lay.theta]
        self.kime.kime_attn_varlen(self.case.qkv if qkv is None else qkv, self.cu, c.max_seqlen, c.heads,
                                   c.kv_heads, lay.window, lay.causal, lay.scale, cs, sn,
                                   out=self.outs[k] if out is None else out, workspace=self.ws,
                                   dev_status=dev_status(self.dev))


class Fp32Run:
    """ModernBERT-base shapes with FP32 qkv: the CUDA-core FP32 path and the
    tensor-core 3xTF32 path (each layer's QK^T and PV as three TF32 products)."""

    def __init__(self, dev):
        import packed_varlen_attention_kime_gb300 as kime
        from packed_varlen_attention_kime_gb300.inputs import varlen_case
        self.kime = kime
        c = self.case = varlen_case("modernbert_base", device=str(dev))
        self.qkv = c.qkv.float()
        self.dev = dev
        self.cu = c.cu_seqlens.to(dev)
        self.tables = {}
        for lay in c.layers:
            if lay.theta not in self.tables:
                cs, sn = kime.kime_rope_tables(lay.theta, c.max_seqlen)
                self.tables[lay.theta] = (cs.to(dev), sn.to(dev))
        self.out = torch.empty((c.total, c.heads * 64), dtype=torch.float32, device=dev)
        n = len(c.lengths)
        self.ws = {p: torch.empty(kime.kime_attn_workspace_bytes(op, n, c.total, c.heads, c.kv_heads),
                                  dtype=torch.uint8, device=dev) for p, op in ((None, 0), ("3xtf32", 4))}
        self.flops = [4 * 64 * c.heads * visible_pairs(c.lengths, l.window, l.causal) for l in c.layers]

    def layer(self, k, precision):
        c, lay = self.case, self.case.layers[k]
        cs, sn = self.tables[lay.theta]
        self.kime.kime_attn_varlen(self.qkv, self.cu, c.max_seqlen, c.heads, c.kv_heads, lay.window, lay.causal,
                                   lay.scale, cs, sn, out=self.out, workspace=self.ws[precision],
                                   dev_status=dev_status(self.dev), precision=precision)


class DecodeRun:
    def __init__(self, dev):
        import packed_varlen_attention_kime_gb300 as kime
        from packed_varlen_attention_kime_gb300.inputs import decode_case
        self.kime = kime
        c = self.case = decode_case(device=str(dev))
        self.dev = dev
        self.pos = c.pos.to(dev)
        cs, sn = kime.kime_rope_tables(c.theta, c.cap)
        self.cs, self.sn = cs.to(dev), sn.to(dev)
        self.out = torch.empty((len(c.pos), c.heads * 64), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(kime.kime_attn_workspace_bytes(1, len(c.pos), 0, c.heads, c.kv_heads, c.cap),
                              dtype=torch.uint8, device=dev)
        keys = (c.pos.long() + 1).sum().item()
        # K and V prefixes read + new rows read + appended rows written + out written
        W = c.qkv_new.shape[1]
        self.bytes = int(keys * c.kv_heads * 64 * 2 * 2 + len(c.pos) * (W * 2 + c.kv_heads * 2 * 128 +
                                                                        c.heads * 64 * 2))
        self.flops = int(4 * 64 * c.heads * keys)

    def step(self):
        c = self.case
        self.kime.kime_decode_step(c.qkv_new, self.pos, c.heads, c.kv_heads, c.k_cache, c.v_cache, c.scale,
                                   self.cs, self.sn, out=self.out, workspace=self.ws, dev_status=dev_status(self.dev))


class ChunkRun:
    """Chunked prefill against the KV cache (SmolLM2 shapes): append the chunks
    and attend, one kime_chunk_step per step (the same positions every step),
    with the workspace of op 5 (prepared rows, the binding's default) or of
    op 2 (the minimum: the kernel that converts its own tiles)."""

    def __init__(self, dev, ws_op=5):
        import packed_varlen_attention_kime_gb300 as kime
        from packed_varlen_attention_kime_gb300.inputs import chunk_case
        self.kime = kime
        c = self.case = chunk_case(device=str(dev))
        self.dev = dev
        self.cu, self.pos = c.cu_seqlens.to(dev), c.pos.to(dev)
        cs, sn = kime.kime_rope_tables(c.theta, c.cap)
        self.cs, self.sn = cs.to(dev), sn.to(dev)
        self.out = torch.empty((c.total, c.heads * 64), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(kime.kime_attn_workspace_bytes(ws_op, len(c.lengths), c.total, c.heads, c.kv_heads,
                                                             c.cap), dtype=torch.uint8, device=dev)
        L = np.array(c.lengths, np.int64)
        P = c.pos.numpy().astype(np.int64)
        keys = int((P + L).sum())                       # cache rows each kv head's prefix spans
        pairs = int((L * P + L * (L + 1) // 2).sum())   # visible (query, key) pairs per head
        W = c.qkv.shape[1]
        # qkv rows read + K/V prefixes read + appended K/V rows written + out written
        self.bytes = int(c.total * W * 2 + keys * c.kv_heads * 256 + c.total * c.kv_heads * 256 +
                         c.total * c.heads * 128)
        self.flops = int(4 * 64 * c.heads * pairs)

    def step(self):
        c = self.case
        self.kime.kime_chunk_step(c.qkv, self.cu, self.pos, c.max_seqlen, c.heads, c.kv_heads, c.k_cache,
                                  c.v_cache, c.scale, self.cs, self.sn, out=self.out, workspace=self.ws,
                                  dev_status=dev_status(self.dev))


class ProjRun:
    """The SmolLM2 prefill fed by its QKV projection (x [T, 576], fused weight
    [960, 576]): fused (kime_attn_varlen_proj: the projection writes the
    prepared rows), projection then attend (kime_qkv_proj writing bf16 qkv,
    then kime_attn_varlen), and the projection alone."""

    def __init__(self, dev):
        import packed_varlen_attention_kime_gb300 as kime
        from packed_varlen_attention_kime_gb300.inputs import proj_case
        self.kime = kime
        c = self.case = proj_case(device=str(dev))
        self.dev = dev
        self.cu = c.cu_seqlens.to(dev)
        cs, sn = kime.kime_rope_tables(c.theta, c.max_seqlen)
        self.cs, self.sn = cs.to(dev), sn.to(dev)
        W = c.w.shape[0]
        self.qkv = torch.empty((c.total, W), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((c.total, c.heads * 64), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(kime.kime_attn_workspace_bytes(3, len(c.lengths), c.total, c.heads, c.kv_heads),
                              dtype=torch.uint8, device=dev)
        self.gemm_flops = 2 * c.total * c.x.shape[1] * W
        self.attn_flops = 4 * 64 * c.heads * visible_pairs(c.lengths, c.window, c.causal)

    def fused(self):
        c = self.case
        self.kime.kime_attn_varlen_proj(c.x, c.w, self.cu, c.max_seqlen, c.heads, c.kv_heads, c.window, c.causal,
                                        c.scale, self.cs, self.sn, out=self.out, workspace=self.ws,
                                        dev_status=dev_status(self.dev))

    def proj(self):
        c = self.case
        self.kime.kime_qkv_proj(c.x, c.w, c.heads, c.kv_heads, out=self.qkv, dev_status=dev_status(self.dev))

    def unfused(self):
        c = self.case
        self.proj()
        self.kime.kime_attn_varlen(self.qkv, self.cu, c.max_seqlen, c.heads, c.kv_heads, c.window, c.causal,
                                   c.scale, self.cs, self.sn, out=self.out, workspace=self.ws,
                                   dev_status=dev_status(self.dev))


def time_fn(fn, n, warmup, flush, stream, events=1):
    """Median and mean ms of fn over n calls, L2 flushed before each; fn gets
    the list of events to record its sub-steps (len events+1)."""
    for _ in range(warmup):
        fn(None)
    torch.cuda.synchronize()
    per = []
    subs = []
    for _ in range(n):
        flush_l2(flush)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(events + 1)]
        ev[0].record(stream)
        fn(ev)
        ev[-1].record(stream)
        torch.cuda.synchronize()
        per.append(ev[0].elapsed_time(ev[-1]))
        subs.append([ev[i].elapsed_time(ev[i + 1]) for i in range(events)])
    return per, subs


def layer_figures(r, k, ms, pk):
    """Throughput and roofline fractions of layer k of a VarlenRun taking ms."""
    tf = r.flops[k] / (ms * 1e-3) / 1e12
    gbs = r.bytes_per_layer / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "tflops": round(tf, 2), "gbs": round(gbs, 1),
            "tc_frac": round(tf / pk["bf16_tflops"], 4), "hbm_frac": round(gbs / pk["hbm_gbs"], 4),
            "roof_frac": round(max(r.flops[k] / (pk["bf16_tflops"] * 1e12),
                                   r.bytes_per_layer / (pk["hbm_gbs"] * 1e9)) / (ms * 1e-3), 4)}


def extra_measurements(dev, flush, stream, pk, reps=200, warmup=20):
    """The other workloads: medians of `reps` flushed repetitions."""
    out = {}
    for name in ("modernbert_base", "smollm2_prefill"):
        r = VarlenRun(name, dev)
        nl = len(r.case.layers)

        def f(ev, r=r, nl=nl):
            for k in range(nl):
                r.layer(k)
                if ev is not None and k + 1 < nl:
                    ev[k + 1].record(stream)
        per, subs = time_fn(f, reps, warmup, flush, stream, events=nl)
        layers = {lay.name: layer_figures(r, k, statistics.median([s[k] for s in subs]), pk)
                  for k, lay in enumerate(r.case.layers)}
        out[name] = {"tokens": r.case.total, "tokens_per_s": round(r.case.total / (statistics.median(per) * 1e-3)),
                     "layers": layers}
        if name == "modernbert_base":
            k = [lay.name for lay in r.case.layers].index("global")
            ms = layers["global"]["ms"]
            ach = r.bytes_per_layer / (ms * 1e-3) / 1e9
            out[name]["roofline"] = {
                "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "traffic": measured_traffic("modernbert_base:global"),
                "kernel": "kime_attn_varlen call, global layer: schedule_kernel + qkv_prep_kernel + "
                          "prefill_rows_kernel; traffic summed over the three",
                "algorithmic_bytes": r.bytes_per_layer, "avg_ms": ms}
        del r
        torch.cuda.empty_cache()
    pr = ProjRun(dev)
    row = {}
    for key, fn in (("fused", pr.fused), ("unfused", pr.unfused), ("proj", pr.proj)):
        per, _ = time_fn(lambda ev, fn=fn: fn(), reps, warmup, flush, stream)
        row[key + "_ms"] = round(statistics.median(per), 4)
    row["proj_tflops"] = round(pr.gemm_flops / (row["proj_ms"] * 1e-3) / 1e12, 1)
    row["fused_tokens_per_s"] = round(pr.case.total / (row["fused_ms"] * 1e-3))
    row["unfused_tokens_per_s"] = round(pr.case.total / (row["unfused_ms"] * 1e-3))
    row["gemm_flops"] = pr.gemm_flops
    row["attn_flops"] = pr.attn_flops
    out["smollm2_proj"] = row
    del pr
    torch.cuda.empty_cache()
    d = DecodeRun(dev)
    per, _ = time_fn(lambda ev: d.step(), reps, warmup, flush, stream)
    ms = statistics.median(per)
    gbs = d.bytes / (ms * 1e-3) / 1e9
    out["smollm2_decode"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm_gbs"], 4),
                             "tokens_per_s": round(len(d.case.pos) / (ms * 1e-3)), "bytes": d.bytes}
    del d
    torch.cuda.empty_cache()
    ch = ChunkRun(dev)
    per, _ = time_fn(lambda ev: ch.step(), reps, warmup, flush, stream)
    ms = statistics.median(per)
    tf = ch.flops / (ms * 1e-3) / 1e12
    out["smollm2_chunk"] = {"ms": round(ms, 4), "tflops": round(tf, 2), "tc_frac": round(tf / pk["bf16_tflops"], 4),
                            "gbs": round(ch.bytes / (ms * 1e-3) / 1e9, 1),
                            "tokens_per_s": round(ch.case.total / (ms * 1e-3)), "flops": ch.flops,
                            "bytes": ch.bytes}
    del ch
    torch.cuda.empty_cache()
    # FP32 qkv: CUDA-core path vs 3xTF32 on the tensor cores.  The tensor work
    # is three TF32 products per useful product; its peak is the measured BF16
    # peak times the nominal TF32 / BF16 ratio (1.1 / 2.25 PFLOP/s dense)
    fr = Fp32Run(dev)
    tf32_peak = pk["bf16_tflops"] * 1.1 / 2.25
    layers = {}
    for k, lay in enumerate(fr.case.layers):
        row = {}
        for prec, key in ((None, "simt"), ("3xtf32", "3xtf32")):
            n = reps if prec else max(reps // 4, 20)  # the CUDA-core path takes ~2 ms a call
            per, _ = time_fn(lambda ev, k=k, prec=prec: fr.layer(k, prec), n, warmup, flush, stream)
            ms = statistics.median(per)
            row[key + "_ms"] = round(ms, 4)
            row[key + "_tflops"] = round(fr.flops[k] / (ms * 1e-3) / 1e12, 2)
        row["3xtf32_tc_frac"] = round(3 * row["3xtf32_tflops"] / tf32_peak, 4)
        layers[lay.name] = row
    out["modernbert_base_fp32"] = {"tokens": fr.case.total, "layers": layers,
                                   "tf32_peak_tflops": round(tf32_peak, 1)}
    del fr
    torch.cuda.empty_cache()
    return out


# ---- CPU oracle leg ----------------------------------------------------------------

def oracle_sample_rate(case, budget_s=15.0, prefix=1024):
    """Oracle throughput (tokens/s over the layer pair) on the first `prefix`
    tokens of the workload's sequences (each a sequence of its own), taken in
    order until about budget_s of CPU work is done."""
    import oracle
    from packed_varlen_attention_kime_gb300.inputs import bf16_bits, cu_from_lengths
    oracle.build()
    x = bf16_bits(case.qkv)
    tabs = {}
    for lay in case.layers:
        c, s = oracle.rope_tables_f32(lay.theta, case.max_seqlen)
        tabs[lay.theta] = (c.astype(np.float64), s.astype(np.float64))
    cores = os.cpu_count() or 1
    tokens, spent, nseq = 0, 0.0, 0
    cu = case.cu_seqlens.numpy()
    while nseq < len(case.lengths) and spent < budget_s:
        a = int(cu[nseq])
        b = min(int(cu[nseq + 1]), a + prefix)
        sub_cu = cu_from_lengths([b - a]).numpy()
        t0 = time.perf_counter()
        for lay in case.layers:
            c, s = tabs[lay.theta]
            oracle.attn_varlen(x[a:b], sub_cu, case.heads, case.kv_heads, lay.window, lay.causal, lay.scale, c, s,
                               nthreads=cores)
        spent += time.perf_counter() - t0
        tokens += b - a
        nseq += 1
    return tokens / spent, cores, (f"the first {prefix} tokens of each of the first {nseq} of {len(case.lengths)} "
                                    f"sequences ({tokens} tokens), both layers")


def oracle_single_core():
    """The oracle on one host core: the whole FP32 tiny batch (ms per call) and
    the decode step's first sequences (ms per sequence, all q heads)."""
    import oracle
    from packed_varlen_attention_kime_gb300.inputs import bf16_bits, decode_case, varlen_case
    oracle.build()
    t = varlen_case("tiny")
    lay = t.layers[0]
    c, s = oracle.rope_tables_f32(lay.theta, t.max_seqlen)
    x = t.qkv.numpy()
    reps = 50
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.attn_varlen(x, t.cu_seqlens.numpy(), t.heads, t.kv_heads, lay.window, lay.causal, lay.scale,
                           c.astype(np.float64), s.astype(np.float64), nthreads=1)
    tiny_ms = (time.perf_counter() - t0) / reps * 1e3
    d = decode_case()
    c, s = oracle.rope_tables_f32(d.theta, d.cap)
    n = 4
    kb, vb = bf16_bits(d.k_cache[:n]), bf16_bits(d.v_cache[:n])
    t0 = time.perf_counter()
    oracle.attn_decode(bf16_bits(d.qkv_new[:n]), d.pos[:n].numpy(), d.heads, d.kv_heads, d.cap, d.scale,
                       c.astype(np.float64), s.astype(np.float64), kb, vb, nthreads=1)
    dec_ms = (time.perf_counter() - t0) / n * 1e3
    return {"cores": 1, "tiny_fp32_ms_per_call": round(tiny_ms, 4),
            "decode_ms_per_seq": round(dec_ms, 3),
            "decode_sample": f"sequences 0-{n - 1} of {len(d.pos)} (keys 0..pos, all {d.heads} q heads)"}


def end_to_end(args, dev, stream, flush, run, world):
    """The headline step end to end through the public API: pinned host qkv ->
    device, both layers, both outputs -> pinned host, every step.  Steps are
    pipelined as a server would run them, with NB sets of device and pinned
    host buffers: step k+1's copy in overlaps step k's layers and step k-1's
    copy out (the link is full duplex), on three streams ordered by events; a
    buffer set is refilled only after the step NB back has finished with it.
    Each step still copies its own inputs in and its results out.  Timed over
    K consecutive steps, the first copy in and the last copy out included."""
    c = run.case
    h_qkv = c.qkv.cpu().pin_memory()
    h_cu = c.cu_seqlens.cpu().to(torch.int32).pin_memory()
    mx = max(c.lengths)
    NB = args.e2e_buffers
    d_qkv = [torch.empty_like(c.qkv) for _ in range(NB)]
    d_cu = [torch.empty_like(h_cu, device=dev) for _ in range(NB)]
    d_out = [[torch.empty_like(o) for o in run.outs] for _ in range(NB)]
    h_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in run.outs] for _ in range(NB)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_cmp = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [torch.cuda.Event() for _ in range(NB)]
    status = dev_status(dev)

    def enqueue(k):
        b = k % NB
        with torch.cuda.stream(s_in):
            if k >= NB:
                s_in.wait_event(ev_cmp[b])  # step k-NB's layers have read this input buffer
            d_qkv[b].copy_(h_qkv, non_blocking=True)
            d_cu[b].copy_(h_cu, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[b])
            if k >= NB:
                s_cmp.wait_event(ev_out[b])  # step k-NB's outputs have left this buffer
            for li, lay in enumerate(c.layers):
                cs, sn = run.tables[lay.theta]
                run.kime.kime_attn_varlen(d_qkv[b], d_cu[b], mx, c.heads, c.kv_heads, lay.window, lay.causal,
                                          lay.scale, cs, sn, out=d_out[b][li], workspace=run.ws,
                                          dev_status=status, stream=s_cmp)
            ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            for h, o in zip(h_out[b], d_out[b]):
                h.copy_(o, non_blocking=True)
            ev_out[b].record(s_out)

    def run_steps(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        for st in (s_in, s_cmp, s_out):
            st.wait_stream(stream)
        for k in range(n):
            enqueue(k)
        for st in (s_in, s_cmp, s_out):
            stream.wait_stream(st)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run_steps(4)  # warm-up (first-call set-up, pinned pages touched)
    n = max(10, args.steps)
    e_ms = max_over_ranks(run_steps(n), dev if world > 1 else None) / n
    # the pipelined steps give the whole batch's bits (every buffer set)
    for k in range(len(c.layers)):
        run.layer(k)
    torch.cuda.synchronize()
    for b in range(NB):
        if not all(torch.equal(x, y) for x, y in zip(d_out[b], run.outs)) or \
                not all(torch.equal(h, o.cpu()) for h, o in zip(h_out[b], run.outs)):
            raise RuntimeError("pipelined end-to-end outputs differ from the whole-batch calls")
    return {"value": round(world * c.total / (e_ms * 1e-3)), "unit": "tokens/s",
            "h2d_bytes_per_step": h_qkv.numel() * 2 + h_cu.numel() * 4,
            "d2h_bytes_per_step": sum(o.numel() * 2 for o in run.outs), "ms_per_step": round(e_ms, 4),
            "pipeline": f"{n} consecutive steps timed together; step k+1's copy in overlaps step k's two layer "
                        f"calls and step k-1's copy out ({NB} buffer sets, three streams); first copy in and last "
                        f"copy out included; no L2 flush between steps: each step's input "
                        f"({h_qkv.numel() * 2 / 1e6:.0f} MB) is larger than L2"}


# ---- main ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (e2e null): profiling runs")
    ap.add_argument("--e2e-buffers", type=int, default=2,
                    help="device and pinned host buffer sets the end-to-end steps rotate through")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s load before the timed steps")
    ap.add_argument("--only", default=None,
                    help="profiling aid: run only WORKLOAD[:LAYER] (modernbert_base, modernbert_large, "
                         "smollm2_proj[:fused|unfused|proj], "
                         "smollm2_prefill, smollm2_decode, smollm2_chunk[:minimal]) for --steps steps and print its "
                         "timings (smollm2_chunk:minimal: the chunk step with the minimal workspace)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.only:
        return only_arm(args, local)

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from __graft_entry__ import build
    build()
    pk, pk_src = peaks()
    stream = torch.cuda.current_stream(dev)
    flush = l2_flush_buffer(dev)
    run = VarlenRun(HEADLINE, dev)
    c = run.case

    def step(ev):
        run.layer(0)
        if ev is not None:
            ev[1].record(stream)
        run.layer(1)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # keep the GPU under the same load for about a second first, so the
        # 100 ms clock samples cover the timed steps and the state they run in
        t_end = time.perf_counter() + (0.0 if args.no_soak else 1.0)
        while time.perf_counter() < t_end:
            for _ in range(20):
                step(None)
            torch.cuda.synchronize()
        per, subs = time_fn(step, args.steps, args.warmup, flush, stream, events=2)
    clocks = clk.summary()
    total_ms = max_over_ranks(sum(per), dev if world > 1 else None)
    ms_step = total_ms / args.steps
    value = world * c.total * args.steps / (total_ms * 1e-3)

    # roofline of the dominant call, the global layer (tensor-bound): its
    # useful FLOPs over the whole call's time (scheduler, row preparation and
    # attention kernel; the attention kernel is most of it, see the launch
    # list in profiles/), against the burst BF16 peak (the call is timed alone
    # between L2 flushes)
    gk = [lay.name for lay in c.layers].index("global")
    lk = [lay.name for lay in c.layers].index("local")
    g_ms = statistics.mean(s[gk] for s in subs)
    l_ms = statistics.mean(s[lk] for s in subs)
    achieved = run.flops[gk] / (g_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / pk["bf16_tflops"], 4),
            "traffic": measured_traffic(f"{HEADLINE}:global"),
            "kernel": "kime_attn_varlen call, ModernBERT-large global layer: schedule_kernel + qkv_prep_kernel + "
                      "prefill_rows_kernel; avg_ms is the whole call, traffic the DRAM bytes of all three",
            "algorithmic_flops": run.flops[gk], "algorithmic_bytes": run.bytes_per_layer,
            "avg_ms": round(g_ms, 5), "peak_source": f"{pk_src} (burst)"}
    flops_step = sum(run.flops)
    tflops = flops_step / (ms_step * 1e-3) / 1e12

    # end to end through the public API, with host buffers (end_to_end)
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, dev, stream, flush, run, world)

    # the same step with a warm L2 (no flush between steps, back to back),
    # labelled: reported beside the cold-L2 value, never as it
    for _ in range(3):
        step(None)
    torch.cuda.synchronize()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(args.steps):
        step(None)
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = w0.elapsed_time(w1) / args.steps
    warm = {"ms_per_step": round(warm_ms, 5), "tokens_per_s": round(world * c.total / (warm_ms * 1e-3)),
            "note": "L2 not flushed between steps (warm); not the headline value"}

    extra = {}
    if not args.no_extra and rank == 0:
        extra = extra_measurements(dev, flush, stream, pk)

    check_status(dev)  # any flagged input error or timed-out wait voids the numbers

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        rate, cores, sample = oracle_sample_rate(VarlenRunCPU(c), args.cpu_budget)
        cpu = {"value": round(rate, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "single_core": oracle_single_core()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "modernbert_large local+global layer pair", "seqs": len(c.lengths),
                       "tokens": c.total, "heads": c.heads, "head_dim": 64,
                       "layers": ["local window 64 theta 1e4", "global full theta 1.6e5"],
                       "l2": "flushed before every timed step: 512 MB write, then a 256 MB read so the lines "
                             "left in L2 are clean", "parallelism": f"dp{world}"},
            "useful_tflops": round(tflops, 3), "tc_frac": round(tflops / pk["bf16_tflops"], 4),
            "layer_ms": {"local": round(l_ms, 5), "global": round(g_ms, 5)},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 6 * args.steps, "warm_l2": warm, "extra": extra,  # 3 per layer: scheduler, row preparation, attention
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def only_arm(args, local):
    """One workload (and optionally one layer) alone: the command ncu captures."""
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from __graft_entry__ import build
    build()
    stream = torch.cuda.current_stream(dev)
    flush = l2_flush_buffer(dev)
    name, _, layer = args.only.partition(":")
    if name in ("smollm2_decode", "smollm2_chunk"):
        d = DecodeRun(dev) if name == "smollm2_decode" else ChunkRun(dev, 2 if layer == "minimal" else 5)
        per, _ = time_fn(lambda ev: d.step(), args.steps, args.warmup, flush, stream)
        check_status(dev)
        print(json.dumps({"only": args.only, "ms": [round(x, 4) for x in per]}))
        return
    if name == "smollm2_proj":  # fused (default), unfused, or the projection alone
        pr = ProjRun(dev)
        fn = {"": pr.fused, "fused": pr.fused, "unfused": pr.unfused, "proj": pr.proj}[layer]
        per, _ = time_fn(lambda ev: fn(), args.steps, args.warmup, flush, stream)
        check_status(dev)
        print(json.dumps({"only": args.only, "ms": [round(x, 4) for x in per]}))
        return
    if name == "modernbert_base_fp32":  # the 3xTF32 path
        fr = Fp32Run(dev)
        ks = [k for k, l in enumerate(fr.case.layers) if not layer or l.name == layer]

        def g(ev):
            for k in ks:
                fr.layer(k, "3xtf32")
        per, _ = time_fn(g, args.steps, args.warmup, flush, stream)
        check_status(dev)
        print(json.dumps({"only": args.only, "layers": [fr.case.layers[k].name for k in ks],
                          "ms": [round(x, 4) for x in per]}))
        return
    r = VarlenRun(name, dev)
    ks = [k for k, l in enumerate(r.case.layers) if not layer or l.name == layer]

    def f(ev):
        for k in ks:
            r.layer(k)
    per, _ = time_fn(f, args.steps, args.warmup, flush, stream)
    check_status(dev)
    print(json.dumps({"only": args.only, "layers": [r.case.layers[k].name for k in ks],
                      "ms": [round(x, 4) for x in per]}))


class VarlenRunCPU:
    """The CPU view of a varlen case for the oracle leg."""

    def __init__(self, case):
        self.qkv = case.qkv.cpu()
        self.cu_seqlens = case.cu_seqlens.cpu()
        self.lengths, self.heads, self.kv_heads = case.lengths, case.heads, case.kv_heads
        self.layers, self.max_seqlen = case.layers, case.max_seqlen


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a bounded sample
    of the headline workload.  Under torchrun only rank 0 runs."""
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    import oracle
    from packed_varlen_attention_kime_gb300.inputs import bf16_bits, cu_from_lengths, varlen_case
    oracle.build()
    case = varlen_case(HEADLINE)
    x = bf16_bits(case.qkv)
    cores = os.cpu_count() or 1
    tabs = {}
    for lay in case.layers:
        cs, sn = oracle.rope_tables_f32(lay.theta, case.max_seqlen)
        tabs[lay.theta] = (cs.astype(np.float64), sn.astype(np.float64))
    cu = case.cu_seqlens.numpy()
    # one step: the first 512 tokens of sequence 0 as a sequence of their own, both layers
    a, b = int(cu[0]), int(cu[0]) + 512
    sub_cu = cu_from_lengths([512]).numpy()

    def step():
        for lay in case.layers:
            cs, sn = tabs[lay.theta]
            oracle.attn_varlen(x[a:b], sub_cu, case.heads, case.kv_heads, lay.window, lay.causal, lay.scale, cs,
                               sn, nthreads=cores)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = (b - a) * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "modernbert_large local+global layer pair",
                       "sample": f"the first {b - a} tokens of sequence 0 of {len(case.lengths)}, both layers, "
                                 "per step"},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"the first {b - a} tokens of sequence 0, both layers, per step"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
