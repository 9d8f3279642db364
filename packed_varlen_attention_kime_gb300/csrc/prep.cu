// prep.cu -- a packed batch's qkv rows prepared once per call for the
// tensor-core attention kernel.
//
// The attention kernel works on units of two 128-row query tiles of one head;
// every unit of a sequence reads all of the sequence's key tiles it can see,
// so inside the kernel each key tile of a long sequence would be rotated
// again for every unit (ceil(L / 256) times under full attention), and the
// RoPE work on the kernel's own warps is what limits short sequences.  This
// pass rotates every query and key once, at its position within its own
// sequence (rotate-half RoPE with the float32 tables; positions restart at
// each sequence, kime-cpu 0.0.17 src/kime_cpu/plan.rs, Step::Rope), scales
// the queries by scale * log2(e), rounds both to f16, and widens every value
// to f16; the attention kernel then loads the prepared rows as they are.  Its
// arithmetic is the attention kernel's own: for the pair (t, t + 32),
// y_t = fma(x_t, c, -(x_{t+32} s)) and y_{t+32} = fma(x_{t+32}, c, x_t s) in
// float32, times the query multiplier for query heads, each rounded once to
// f16, so the attention results are the same bits with or without this pass.
//
// Output: rows [total, W] f16 in the qkv layout (W = 64 * (heads + 2 *
// kv_heads)).  One warp per row; lane q of a round holds the 16-byte chunk q
// of the row (8 elements of head q / 8) and swaps it with lane q ^ 4, which
// holds the other half of the rotation pairs.
#include "kime_common.cuh"

namespace kime {

namespace {

// rows (one warp each) per CTA: small CTAs fill the SMs more evenly
// (ModernBERT-base local, means of 400 calls: 0.0797 ms with 2, 0.0812 with
// 4, 0.0810 with 8 and 0.0823 with 16; the other layers level)
constexpr int kPrepWarps = 2;

// kBatch: rounds of 16-byte chunks per lane loaded before any is used -- 4
// for rows of at least 128 query and key chunks (per local / global call,
// ModernBERT-large 0.1649 / 0.9697 ms against 0.169 / 0.9739 with 2, and
// 0.1833 / 0.9882 with 8 at 94 registers a thread; ModernBERT-base, means of
// 400 calls, 0.0824 / 0.0923 against 0.0834 / 0.0938 with 2, and 2 against 1
// 0.0829 / 0.0932 against 0.0850 / 0.0952 in medians), 1 for narrower rows,
// where the longer code costs more than it saves (SmolLM2 prefill: 0.0645 ms
// against 0.0666 with 2 or 4).
template <int kBatch>
__global__ void __launch_bounds__(32 * kPrepWarps)
    qkv_prep_kernel(const uint16_t* __restrict__ qkv, const int32_t* __restrict__ cu, int n_seqs, int total,
                    int heads, int kv_heads, float qmul, const float* __restrict__ cos_t,
                    const float* __restrict__ sin_t, int rope_len, uint16_t* __restrict__ out,
                    int32_t* dev_status) {
  // The attention kernel after this one may launch as soon as every CTA of
  // this grid has started: it sets itself up while the last CTAs run and
  // waits for this grid's results before reading them.
  griddep_launch_dependents();
  const int j = blockIdx.x * kPrepWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (j >= total) {
    griddep_wait();
    return;
  }
  // the sequence owning row j: the largest s with cu[s] <= j; its position there
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= j) lo = mid;
    else hi = mid - 1;
  }
  const int pos = j - __ldg(cu + lo);
  // a row outside [0, rope_len) belongs to no valid sequence (the scheduler
  // reports the bad cu_seqlens and skips it): converted without rotation
  const bool rot = pos >= 0 && pos < rope_len;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  const uint4* src = reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(j) * W);
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(j) * W);
  const int nrot = (heads + kv_heads) * (kHead / 8);  // 16-byte chunks of the row's queries and keys
  const int nall = (heads + 2 * kv_heads) * (kHead / 8);
  float big = 0.f;  // largest magnitude rounded to f16 in this row (an operand beyond kF16Max saturates)
  const float* crow = cos_t + static_cast<size_t>(rot ? pos : 0) * kHalf;
  const float* srow = sin_t + static_cast<size_t>(rot ? pos : 0) * kHalf;
  // every chunk of a lane sits at the same place in its head (lane mod 8), so
  // its rotation pairs' table entries are the same in every round: the
  // four-deep variant loads them once (ModernBERT-base, means of 400 calls,
  // 0.0814 / 0.0912 ms per local / global call against 0.0829 / 0.0926), the
  // narrow rows' variant each round (SmolLM2 prefill: 0.0666 against 0.0684
  // with them loaded once)
  float4 c0h, c1h, s0h, s1h;
  if constexpr (kBatch >= 4) {
    const int th = (lane & 3) * 8;
    c0h = __ldg(reinterpret_cast<const float4*>(crow + th));
    c1h = __ldg(reinterpret_cast<const float4*>(crow + th + 4));
    s0h = __ldg(reinterpret_cast<const float4*>(srow + th));
    s1h = __ldg(reinterpret_cast<const float4*>(srow + th + 4));
  }
  // queries and keys: every lane takes part in each round (the partner
  // exchange needs the whole warp); chunks q and q ^ 4 are both in range or
  // both out of it
  // kBatch rounds' loads are issued before any of them is used, so a warp
  // keeps that many of the row's chunks per lane in flight.
    for (int q0 = 0; q0 < nrot; q0 += 32 * kBatch) {
    uint4 xs[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int q = q0 + 32 * k + lane;
      xs[k] = q < nrot ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (q0 + 32 * k >= nrot) break;  // (uniform over the warp)
      const int q = q0 + 32 * k + lane;
      const bool in = q < nrot;
      const uint4 x = xs[k];
      uint4 y;
      y.x = __shfl_xor_sync(0xffffffffu, x.x, 4);
      y.y = __shfl_xor_sync(0xffffffffu, x.y, 4);
      y.z = __shfl_xor_sync(0xffffffffu, x.z, 4);
      y.w = __shfl_xor_sync(0xffffffffu, x.w, 4);
      if (!in) continue;
      const int a = q & 7;                                 // chunk within the head: 0..3 low half, 4..7 high half
      const float mul = (q >> 3) < heads ? qmul : 1.f;     // query heads carry scale * log2(e)
      uint4 o;
      if (rot) {
        float4 c0, c1, s0, s1;
        if constexpr (kBatch >= 4) {
          c0 = c0h;
          c1 = c1h;
          s0 = s0h;
          s1 = s1h;
        } else {
          const int t0 = (a & 3) * 8;  // pair index of the chunk's first element
          c0 = __ldg(reinterpret_cast<const float4*>(crow + t0));
          c1 = __ldg(reinterpret_cast<const float4*>(crow + t0 + 4));
          s0 = __ldg(reinterpret_cast<const float4*>(srow + t0));
          s1 = __ldg(reinterpret_cast<const float4*>(srow + t0 + 4));
        }
        const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
        uint32_t ow[4];
  #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16lo(xw[e]), x1 = bf16hi(xw[e]), p0 = bf16lo(yw[e]), p1 = bf16hi(yw[e]);
          float r0, r1;
          if (a < 4) {  // y_t = x_t c - x_{t+32} s
            r0 = __fmaf_rn(x0, cc[2 * e], -__fmul_rn(p0, ss[2 * e]));
            r1 = __fmaf_rn(x1, cc[2 * e + 1], -__fmul_rn(p1, ss[2 * e + 1]));
          } else {      // y_{t+32} = x_{t+32} c + x_t s
            r0 = __fmaf_rn(x0, cc[2 * e], __fmul_rn(p0, ss[2 * e]));
            r1 = __fmaf_rn(x1, cc[2 * e + 1], __fmul_rn(p1, ss[2 * e + 1]));
          }
          big = fmax3(big, fabsf(r0 * mul), fabsf(r1 * mul));
          ow[e] = pack_f16x2(r0 * mul, r1 * mul);
        }
        o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      } else {  // a row of no valid sequence: converted only (its range is not checked)
        o = make_uint4(pack_f16x2(bf16lo(x.x), bf16hi(x.x)), pack_f16x2(bf16lo(x.y), bf16hi(x.y)),
                       pack_f16x2(bf16lo(x.z), bf16hi(x.z)), pack_f16x2(bf16lo(x.w), bf16hi(x.w)));
      }
      dst[q] = o;
    }
  }
  // values: widened to f16 (kBatch loads in flight per lane)
  for (int q0 = nrot; q0 < nall; q0 += 32 * kBatch) {
    uint4 xs[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int q = q0 + 32 * k + lane;
      xs[k] = q < nall ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int q = q0 + 32 * k + lane;
      if (q >= nall) break;
      const uint4 x = xs[k];
      big = fmax3(big, fmax3(fabsf(bf16lo(x.x)), fabsf(bf16hi(x.x)), fabsf(bf16lo(x.y))),
                  fmax3(fabsf(bf16hi(x.y)), fmax3(fabsf(bf16lo(x.z)), fabsf(bf16hi(x.z)), fabsf(bf16lo(x.w))),
                        fabsf(bf16hi(x.w))));
      dst[q] = make_uint4(pack_f16x2(bf16lo(x.x), bf16hi(x.x)), pack_f16x2(bf16lo(x.y), bf16hi(x.y)),
                          pack_f16x2(bf16lo(x.z), bf16hi(x.z)), pack_f16x2(bf16lo(x.w), bf16hi(x.w)));
    }
  }
  if (__any_sync(0xffffffffu, rot && big > kF16Max) && lane == 0) report(dev_status, ST_RANGE);
  // this pass runs beside the scheduler (it reads none of its output); it
  // ends only after the scheduler has, so the attention kernel, which waits
  // for this pass, also finds the scheduler's lists complete
  griddep_wait();
}

}  // namespace

cudaError_t launch_qkv_prep(const void* qkv, const int32_t* cu, int n_seqs, int total, int heads, int kv_heads,
                            float scale, const float* cos_t, const float* sin_t, int rope_len, void* out,
                            int32_t* dev_status, cudaStream_t st) {
  // launched with programmatic stream serialization: it starts while the
  // scheduler (which lets dependents start at once) still runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((total + kPrepWarps - 1) / kPrepWarps);
  cfg.blockDim = dim3(32 * kPrepWarps);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float qmul = scale * 1.4426950408889634f;
  const uint16_t* src = static_cast<const uint16_t*>(qkv);
  uint16_t* dst = static_cast<uint16_t*>(out);
  if ((heads + kv_heads) * (kHead / 8) >= 128)  // chunks of a row's queries and keys
    return cudaLaunchKernelEx(&cfg, qkv_prep_kernel<4>, src, cu, n_seqs, total, heads, kv_heads, qmul, cos_t, sin_t,
                              rope_len, dst, dev_status);
  return cudaLaunchKernelEx(&cfg, qkv_prep_kernel<1>, src, cu, n_seqs, total, heads, kv_heads, qmul, cos_t, sin_t,
                            rope_len, dst, dev_status);
}

}  // namespace kime
