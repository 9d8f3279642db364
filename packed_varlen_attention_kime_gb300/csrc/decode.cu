// decode.cu -- in-place KV-cache append and single-token split-KV decode.
//
// Append (ffai-argus 0.7.3 src/text.rs, KvAppend): the new token's k heads,
// RoPE'd at position pos[s], and its v heads are written into row pos[s] of
// caches laid out [n_seqs, kv_heads, cap, 64] (bf16); for one (s, kv head)
// the used prefix is one contiguous run of rows.  The position is checked
// against cap (and the RoPE table) before anything is written.
//
// Decode (ffai-argus CausalSoftmax with q_len 1 and offset k_len-1): the new
// token's q head h, RoPE'd at pos[s], attends to cache rows 0..=pos[s] of kv
// head h / (heads/kv_heads), all heads of one kv group together (the GQA fold
// of TextTower::block: the cache is never expanded per q head).
//
// Split-KV: one CTA per (key chunk of 256, kv head, sequence).  The chunk's K
// and V rows arrive by two 1-D bulk copies into shared memory; 8 threads share
// a key (8 dims each), so scores need a 3-step shuffle reduction.  Each CTA
// reduces its chunk to (m, l, o[64]) per q head (base-2 logits); the last CTA
// of a (sequence, kv head) to finish -- found with an atomic ticket, no waiting
// -- merges the chunks: m = max m_c, l = sum l_c 2^(m_c-m), o = sum o_c 2^(m_c-m) / l.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kDecThreads = 128;
constexpr int kGroups = kDecThreads / 8;        // keys processed at once
constexpr int kKeysPerThread = kDecChunk / kGroups;
constexpr int kPartialFloats = 68;               // m, l, o[64], 2 pad
constexpr uint32_t kDecSmem = 2 * kDecChunk * kHead * 2 + 64;

__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const uint16_t* __restrict__ qkv_new, const int32_t* __restrict__ pos, int heads,
                     int kv_heads, int cap, const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                     int rope_len, uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                     int32_t* dev_status) {
  const int s = blockIdx.x;
  const int P = pos[s];
  if (P < 0 || P >= cap || P >= rope_len) {
    if (threadIdx.x == 0) report(dev_status, ST_BAD_POS);
    return;
  }
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  const uint16_t* row = qkv_new + static_cast<size_t>(s) * W;
  for (int e = threadIdx.x; e < kv_heads * kHalf; e += blockDim.x) {
    const int g = e / kHalf, t = e % kHalf;
    const uint16_t* xk = row + (heads + g) * kHead;
    const float a = __uint_as_float(static_cast<uint32_t>(xk[t]) << 16);
    const float b = __uint_as_float(static_cast<uint32_t>(xk[t + kHalf]) << 16);
    float ya, yb;
    rope_pair(a, b, cos_t[static_cast<size_t>(P) * kHalf + t], sin_t[static_cast<size_t>(P) * kHalf + t], ya, yb);
    const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
    const uint32_t w = pack_bf16x2(ya, yb);
    k_cache[dst + t] = static_cast<uint16_t>(w & 0xffffu);
    k_cache[dst + t + kHalf] = static_cast<uint16_t>(w >> 16);
  }
  for (int e = threadIdx.x; e < kv_heads * kHead; e += blockDim.x) {
    const int g = e / kHead, t = e % kHead;
    const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
    v_cache[dst + t] = row[(heads + kv_heads + g) * kHead + t];
  }
}

template <int G>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const uint16_t* __restrict__ qkv_new, const int32_t* __restrict__ pos, int heads, int kv_heads,
                  int cap, float scale_log2, const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                  int rope_len, const uint16_t* __restrict__ k_cache, const uint16_t* __restrict__ v_cache,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ partials, int32_t* __restrict__ tickets,
                  int max_chunks, int32_t* dev_status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vs = Ks + kDecChunk * kHead;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * kDecChunk * kHead * 2);
  __shared__ int s_last;

  const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x;
  const int P = pos[s];
  if (P < 0 || P >= cap || P >= rope_len) {
    if (c == 0 && g == 0 && tid == 0) report(dev_status, ST_BAD_POS);
    return;
  }
  const int n_keys = P + 1;
  const int n_c = (n_keys + kDecChunk - 1) / kDecChunk;
  if (c >= n_c) return;
  const int j0 = c * kDecChunk;
  const int nk = min(kDecChunk, n_keys - j0);
  const size_t base = ((static_cast<size_t>(s) * kv_heads + g) * cap + j0) * kHead;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, 2u * nk * kHead * 2);
    bulk_load(Ks, k_cache + base, nk * kHead * 2, bar);
    bulk_load(Vs, v_cache + base, nk * kHead * 2, bar);
  }

  // q heads of this kv group, RoPE'd at P, this thread's 8 dims, pre-multiplied
  // by scale * log2(e).
  const int lane8 = tid & 7, grp = tid >> 3;
  const int d0 = lane8 * 8;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  float q[G][8];
  {
    const int tb = d0 & (kHalf - 1);
    const float* cp = cos_t + static_cast<size_t>(P) * kHalf + tb;
    const float* sp = sin_t + static_cast<size_t>(P) * kHalf + tb;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const uint16_t* xq = qkv_new + static_cast<size_t>(s) * W + (g * G + hh) * kHead;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = tb + e;
        const float a = __uint_as_float(static_cast<uint32_t>(xq[t]) << 16);
        const float b = __uint_as_float(static_cast<uint32_t>(xq[t + kHalf]) << 16);
        float ya, yb;
        rope_pair(a, b, cp[e], sp[e], ya, yb);
        q[hh][e] = (d0 < kHalf ? ya : yb) * scale_log2;
      }
    }
  }
  __syncthreads();  // barrier initialised before anyone waits on it
  const bool ok = mbar_wait(bar, 0);
  if (__syncthreads_or(!ok)) {
    // The copies did not land in time: report, give them one more bounded
    // wait so the shared memory outlives them, and leave the chunk undone.
    if (tid == 0) {
      report(dev_status, ST_TIMEOUT);
      mbar_wait(bar, 0);
    }
    return;
  }

  // Scores of this thread's keys (grp, grp + 16, ...).
  float sc[G][kKeysPerThread];
#pragma unroll
  for (int it = 0; it < kKeysPerThread; ++it) {
    const int kk = grp + it * kGroups;
    float part[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) part[hh] = 0.f;
    if (kk < nk) {
      const uint4 kw = *reinterpret_cast<const uint4*>(Ks + kk * kHead + d0);
      const float kf[8] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y),
                           bf16lo(kw.z), bf16hi(kw.z), bf16lo(kw.w), bf16hi(kw.w)};
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < 8; ++e) part[hh] = fmaf(q[hh][e], kf[e], part[hh]);
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float v = part[hh];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      sc[hh][it] = kk < nk ? v : -INFINITY;
    }
  }
  float m[G], l[G], o[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float mx = -INFINITY;
#pragma unroll
    for (int it = 0; it < kKeysPerThread; ++it) mx = fmaxf(mx, sc[hh][it]);
    m[hh] = mx;
    l[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[hh][e] = 0.f;
  }
#pragma unroll
  for (int it = 0; it < kKeysPerThread; ++it) {
    const int kk = grp + it * kGroups;
    if (kk >= nk) continue;
    const uint4 vw = *reinterpret_cast<const uint4*>(Vs + kk * kHead + d0);
    const float vf[8] = {bf16lo(vw.x), bf16hi(vw.x), bf16lo(vw.y), bf16hi(vw.y),
                         bf16lo(vw.z), bf16hi(vw.z), bf16lo(vw.w), bf16hi(vw.w)};
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float p = fast_exp2(sc[hh][it] - m[hh]);
      l[hh] += p;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[hh][e] = fmaf(p, vf[e], o[hh][e]);
    }
  }
  __syncthreads();  // K/V consumed; reuse the K area for the cross-group merge

  float* red_o = reinterpret_cast<float*>(smem);          // [kGroups][G][64]
  float* red_m = red_o + kGroups * G * kHead;             // [kGroups][G]
  float* red_l = red_m + kGroups * G;                     // [kGroups][G]
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
#pragma unroll
    for (int e = 0; e < 8; ++e) red_o[(grp * G + hh) * kHead + d0 + e] = o[hh][e];
    if (lane8 == 0) {
      red_m[grp * G + hh] = m[hh];
      red_l[grp * G + hh] = l[hh];
    }
  }
  __syncthreads();

  const bool single = n_c == 1;
  float* part = partials + ((static_cast<size_t>(s) * kv_heads + g) * max_chunks + c) * G * kPartialFloats;
  for (int e = tid; e < G * kHead; e += kDecThreads) {
    const int hh = e / kHead, d = e % kHead;
    float M = -INFINITY;
#pragma unroll
    for (int gr = 0; gr < kGroups; ++gr) M = fmaxf(M, red_m[gr * G + hh]);
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int gr = 0; gr < kGroups; ++gr) {
      const float w = fast_exp2(red_m[gr * G + hh] - M);
      Lsum = fmaf(red_l[gr * G + hh], w, Lsum);
      O = fmaf(red_o[(gr * G + hh) * kHead + d], w, O);
    }
    if (single) {
      out[static_cast<size_t>(s) * heads * kHead + (g * G + hh) * kHead + d] = __float2bfloat16_rn(O / Lsum);
    } else {
      part[hh * kPartialFloats + 2 + d] = O;
      if (d == 0) {
        part[hh * kPartialFloats] = M;
        part[hh * kPartialFloats + 1] = Lsum;
      }
    }
  }
  if (single) return;

  // Publish this chunk; the last CTA of (s, g) to arrive merges all chunks.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&tickets[s * kv_heads + g], 1) == n_c - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* all = partials + (static_cast<size_t>(s) * kv_heads + g) * max_chunks * G * kPartialFloats;
  for (int e = tid; e < G * kHead; e += kDecThreads) {
    const int hh = e / kHead, d = e % kHead;
    float M = -INFINITY;
    for (int cc = 0; cc < n_c; ++cc) M = fmaxf(M, __ldcg(all + (cc * G + hh) * kPartialFloats));
    float Lsum = 0.f, O = 0.f;
    for (int cc = 0; cc < n_c; ++cc) {
      const float* pc = all + (cc * G + hh) * kPartialFloats;
      const float w = fast_exp2(__ldcg(pc) - M);
      Lsum = fmaf(__ldcg(pc + 1), w, Lsum);
      O = fmaf(__ldcg(pc + 2 + d), w, O);
    }
    out[static_cast<size_t>(s) * heads * kHead + (g * G + hh) * kHead + d] = __float2bfloat16_rn(O / Lsum);
  }
}

template <int G>
cudaError_t launch_decode_g(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                            float scale, const float* cos_t, const float* sin_t, int rope_len, const void* k_cache,
                            const void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const int max_chunks = dec_chunks_for(cap);
  int32_t* tickets = static_cast<int32_t*>(ws);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                             align_up(static_cast<size_t>(n_seqs) * kv_heads * 4, 256));
  cudaError_t e = cudaMemsetAsync(tickets, 0, static_cast<size_t>(n_seqs) * kv_heads * 4, st);
  if (e != cudaSuccess) return e;
  dim3 grid(max_chunks, kv_heads, n_seqs);
  decode_kernel<G><<<grid, kDecThreads, kDecSmem, st>>>(
      static_cast<const uint16_t*>(qkv_new), pos, heads, kv_heads, cap, scale * 1.4426950408889634f, cos_t, sin_t,
      rope_len, static_cast<const uint16_t*>(k_cache), static_cast<const uint16_t*>(v_cache),
      static_cast<__nv_bfloat16*>(out), partials, tickets, max_chunks, dev_status);
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(int n_seqs, int heads, int kv_heads, int cap) {
  const size_t tickets = align_up(static_cast<size_t>(n_seqs) * kv_heads * 4, 256);
  const size_t parts = static_cast<size_t>(n_seqs) * kv_heads * dec_chunks_for(cap) * (heads / kv_heads) *
                       kPartialFloats * sizeof(float);
  return tickets + parts;
}

cudaError_t launch_kv_append(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                             const float* cos_t, const float* sin_t, int rope_len, void* k_cache, void* v_cache,
                             int32_t* dev_status, cudaStream_t st) {
  kv_append_kernel<<<n_seqs, kAppendThreads, 0, st>>>(static_cast<const uint16_t*>(qkv_new), pos, heads, kv_heads,
                                                      cap, cos_t, sin_t, rope_len, static_cast<uint16_t*>(k_cache),
                                                      static_cast<uint16_t*>(v_cache), dev_status);
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                          float scale, const float* cos_t, const float* sin_t, int rope_len, const void* k_cache,
                          const void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st) {
  switch (heads / kv_heads) {
#define KIME_G(N) \
  case N:         \
    return launch_decode_g<N>(qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t, rope_len, k_cache, v_cache, out, ws, dev_status, st);
    KIME_G(1) KIME_G(2) KIME_G(3) KIME_G(4) KIME_G(5) KIME_G(6) KIME_G(7) KIME_G(8)
#undef KIME_G
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kime
