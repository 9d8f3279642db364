// varlen_f32.cu -- packed variable-length attention for FP32 qkv / FP32 out
// on the CUDA cores (FP32 FMA).
//
// Same schedule, tile classification and semantics as the tensor-core BF16
// kernel; it exists because FP32 inputs must keep FP32 accuracy (max abs error
// 1e-5 against the FP64 oracle), which neither BF16 nor single TF32
// tensor-core operands can give (the tensor-core alternative, three TF32
// products per product, is tf32x3.cu).  kime-cuda 0.0.3 (src/plan.rs, Step::Attention) likewise
// keeps attention's qkv in FP32 (fn types: FP16 rounding of q and k moves
// ModernBERT's softmax).
//
// Persistent CTAs of 128 threads take (pair, head) units from the schedule.
// Thread t owns query row q0 + t: its RoPE'd q and its output accumulator live
// in registers; each visited key tile is RoPE'd once into shared memory with V,
// and the online softmax runs over 16-key chunks, skipping masked keys.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 16;
static_assert(kChunk <= 32, "one visibility bit per key of a chunk");

__device__ __forceinline__ bool visible(int i, int j, int L, int causal, int window) {
  if (j >= L) return false;
  if (causal && j > i) return false;
  if (window >= 0 && abs(i - j) > window) return false;
  return true;
}

// Load one 64-wide head of row `row`, column `col0`, and rotate it at position p.
__device__ __forceinline__ void load_rotated(const float* __restrict__ qkv, size_t W, int row, int col0, int p,
                                             const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                                             float (&y)[kHead]) {
  const float* x = qkv + static_cast<size_t>(row) * W + col0;
  const float* c = cos_t + static_cast<size_t>(p) * kHalf;
  const float* s = sin_t + static_cast<size_t>(p) * kHalf;
#pragma unroll
  for (int t = 0; t < kHalf; ++t) {
    float a = __ldg(x + t), b = __ldg(x + t + kHalf);
    rope_pair(a, b, __ldg(c + t), __ldg(s + t), y[t], y[t + kHalf]);
  }
}

// Output element stores: FP32, or FP32 rounded once to FP16 / BF16 (nearest
// even) for the mixed-precision variant (FP32 qkv, 16-bit out).
__device__ __forceinline__ void store4(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(__half* dst, float a, float b, float c, float d) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_f16x2(a, b), pack_f16x2(c, d));
}
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float a, float b, float c, float d) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads)
    varlen_f32_kernel(const float* __restrict__ qkv, int heads, int kv_heads, int window, int causal, float scale,
                      const float* __restrict__ cos_t, const float* __restrict__ sin_t, OutT* __restrict__ out,
                      WsHeader* hdr, const Pair* __restrict__ pairs) {
  extern __shared__ float4 smem_f4[];
  float(*Ks)[kHead] = reinterpret_cast<float(*)[kHead]>(smem_f4);
  float(*Vs)[kHead] = reinterpret_cast<float(*)[kHead]>(reinterpret_cast<float*>(smem_f4) + kBN * kHead);
  __shared__ int s_unit;

  const int tid = threadIdx.x;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  const int G = heads / kv_heads;
  griddep_wait();  // the schedule written by the kernel before this one
  const int n_units = hdr->n_pairs * heads;

  for (;;) {
    if (tid == 0) s_unit = atomicAdd(&hdr->next_unit, 1);
    __syncthreads();
    const int u = s_unit;
    if (u >= n_units) break;
    const Pair pr = pairs[u / heads];
    const int h = u % heads, g = h / G;
    const int i = pr.qt * kBM + tid;
    const bool valid = i < pr.L;
    const int kcol = (heads + g) * kHead, vcol = (heads + kv_heads + g) * kHead;

    float q[kHead], o[kHead];
    float m = kNone, l = 0.f;  // kNone: no visible key yet (finite, below every logit)
#pragma unroll
    for (int d = 0; d < kHead; ++d) o[d] = 0.f;
    if (valid) load_rotated(qkv, W, pr.row0 + i, h * kHead, i, cos_t, sin_t, q);

    for (int kt = pr.kt_begin; kt < pr.kt_end; ++kt) {
      const int k0 = kt * kBN;
      __syncthreads();  // the previous tile is consumed
      {
        const int j = k0 + tid;
        if (j < pr.L) {
          float kr[kHead];
          load_rotated(qkv, W, pr.row0 + j, kcol, j, cos_t, sin_t, kr);
          const float* vr = qkv + static_cast<size_t>(pr.row0 + j) * W + vcol;
#pragma unroll
          for (int d = 0; d < kHead; ++d) {
            Ks[tid][d] = kr[d];
            Vs[tid][d] = __ldg(vr + d);
          }
        } else {
#pragma unroll
          for (int d = 0; d < kHead; ++d) Ks[tid][d] = Vs[tid][d] = 0.f;
        }
      }
      __syncthreads();
      if (!valid) continue;
      const bool full = kt >= pr.full_begin && kt < pr.full_end;
      for (int c = 0; c < kBN; c += kChunk) {
        // scores of the visible keys only; masked keys are skipped in the
        // maximum and get probability 0 (no -inf is formed)
        float sc[kChunk];
        uint32_t vis = 0;
        float cmax = kNone;
#pragma unroll
        for (int jj = 0; jj < kChunk; ++jj) {
          const int j = k0 + c + jj;
          sc[jj] = 0.f;
          if (full || visible(i, j, pr.L, causal, window)) {
            float acc = 0.f;
#pragma unroll
            for (int d = 0; d < kHead; ++d) acc = fmaf(q[d], Ks[c + jj][d], acc);
            sc[jj] = acc * scale;
            vis |= 1u << jj;
            cmax = fmaxf(cmax, sc[jj]);
          }
        }
        if (vis == 0) continue;
        const float m_new = fmaxf(m, cmax);
        const float alpha = expf(m - m_new);  // 0 while m is kNone (l and o are 0 then)
        l *= alpha;
#pragma unroll
        for (int d = 0; d < kHead; ++d) o[d] *= alpha;
#pragma unroll
        for (int jj = 0; jj < kChunk; ++jj) {
          float p = expf(sc[jj] - m_new);
          if (!((vis >> jj) & 1u)) p = 0.f;
          l += p;
#pragma unroll
          for (int d = 0; d < kHead; ++d) o[d] = fmaf(p, Vs[c + jj][d], o[d]);
        }
        m = m_new;
      }
    }
    if (valid) {
      OutT* dst = out + static_cast<size_t>(pr.row0 + i) * heads * kHead + h * kHead;
      const float inv = 1.f / l;
#pragma unroll
      for (int d = 0; d < kHead; d += 4) store4(dst + d, o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
    }
    __syncthreads();  // s_unit is rewritten at the top
  }
}

template <typename OutT>
cudaError_t launch_f32_as(const float* qkv, int heads, int kv_heads, int window, int causal, float scale,
                          const float* cos_t, const float* sin_t, OutT* out, void* ws, cudaStream_t st) {
  static int configured[64] = {0};
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int smem = 2 * kBN * kHead * static_cast<int>(sizeof(float));
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(varlen_f32_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  const Pair* pairs = reinterpret_cast<const Pair*>(static_cast<char*>(ws) + sizeof(WsHeader));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms * 2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, varlen_f32_kernel<OutT>, qkv, heads, kv_heads, window, causal, scale, cos_t, sin_t,
                            out, hdr, pairs);
}

}  // namespace

cudaError_t launch_varlen_f32(const float* qkv, const int32_t* cu, int n_seqs, int total, int heads, int kv_heads,
                              int window, int causal, float scale, const float* cos_t, const float* sin_t,
                              void* out, int out_kind, void* ws, int max_pairs, int32_t* dev_status,
                              cudaStream_t st) {
  (void)cu; (void)n_seqs; (void)total; (void)max_pairs; (void)dev_status;
  if (out_kind == 1)
    return launch_f32_as(qkv, heads, kv_heads, window, causal, scale, cos_t, sin_t, static_cast<__half*>(out), ws, st);
  if (out_kind == 2)
    return launch_f32_as(qkv, heads, kv_heads, window, causal, scale, cos_t, sin_t, static_cast<__nv_bfloat16*>(out),
                         ws, st);
  return launch_f32_as(qkv, heads, kv_heads, window, causal, scale, cos_t, sin_t, static_cast<float*>(out), ws, st);
}

}  // namespace kime
