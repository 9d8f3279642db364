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
// Split-KV: one CTA per (two chunks of 128 keys, kv head, sequence); CTAs
// past pos[s] exit at once.  Each chunk's K and V rows arrive by two 1-D bulk
// copies into their own shared-memory stage -- all issued at the start, so the
// second chunk lands while the first is computed and q is rotated.  8 threads share
// a key (8 dims each), so scores need a 3-step shuffle reduction; all G q heads
// of the kv group are done together, with an online softmax across the two
// chunks.  Each CTA reduces its keys to (m, l, o[64]) per q head (base-2
// logits); the last CTA of a (sequence, kv head) to finish -- found with an
// atomic ticket, no waiting -- merges the parts:
// m = max m_c, l = sum l_c 2^(m_c-m), o = sum o_c 2^(m_c-m) / l.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kDecThreads = 128;
constexpr int kGroups = kDecThreads / 8;        // keys processed at once (8 threads per key)
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kKeysPerThread = kDecChunk / kGroups;
constexpr uint32_t kStageBytes = 2 * kDecChunk * kHead * 2;  // K and V of one chunk
constexpr int kPartialFloats = 68;               // m, l, o[64], 2 pad

constexpr int kDecPer = 2;  // chunks per CTA: the second one's copies land while the first is computed

template <int G>
constexpr uint32_t dec_smem_bytes() {
  return kDecPer * kStageBytes + ((kDecWarps * G * kHead + 2 * kDecWarps * G) * 4 + 15) / 16 * 16 + 8 * kDecPer;
}

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

// kAppend: the CTA whose chunk holds row pos[s] also performs the KV append of
// kv_append_kernel for its kv head (the same float32 rotation and rounding),
// writes the row to the caches and patches its shared-memory copy, so append
// and attention take one launch.  No other CTA reads that row.
template <int G, bool kAppend>
__global__ void __launch_bounds__(kDecThreads, G > 4 ? 2 : 3)
    decode_kernel(const uint16_t* __restrict__ qkv_new, const int32_t* __restrict__ pos, int n_seqs, int heads,
                  int kv_heads, int cap, float scale_log2, const float* __restrict__ cos_t,
                  const float* __restrict__ sin_t, int rope_len, uint16_t* __restrict__ k_cache,
                  uint16_t* __restrict__ v_cache, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ partials, int32_t* __restrict__ tickets, int max_chunks, int32_t* dev_status) {
  extern __shared__ __align__(128) uint8_t smem[];
  // [K | V of chunk A][K | V of chunk B][merge buffers][2 mbarriers]
  float* red_o = reinterpret_cast<float*>(smem + kDecPer * kStageBytes);  // [warps][G][64]
  float* red_m = red_o + kDecWarps * G * kHead;                            // [warps][G]
  float* red_l = red_m + kDecWarps * G;                                    // [warps][G]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kDecPer * kStageBytes +
                                              ((kDecWarps * G * kHead + 2 * kDecWarps * G) * 4 + 15) / 16 * 16);
  __shared__ int s_last;
  (void)n_seqs;

  const int pc = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, lane8 = tid & 7, grp = tid >> 3, d0 = lane8 * 8;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  const int P = __ldg(pos + s);
  if (P < 0 || P >= cap || P >= rope_len) {
    if (pc == 0 && g == 0 && tid == 0) report(dev_status, ST_BAD_POS);
    return;
  }
  const int n_c = (P + 1 + kDecChunk - 1) / kDecChunk;  // chunks of keys 0..=P
  const int n_parts = (n_c + kDecPer - 1) / kDecPer;      // CTAs for this (s, g)
  if (pc >= n_parts) return;
  const int c_first = pc * kDecPer, n_here = min(kDecPer, n_c - c_first);
  if (tid == 0) {
    for (int i = 0; i < kDecPer; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
    for (int i = 0; i < n_here; ++i) {
      const int c = c_first + i, nk = min(kDecChunk, P + 1 - c * kDecChunk);
      const size_t base =
          ((static_cast<size_t>(s) * kv_heads + g) * cap + static_cast<size_t>(c) * kDecChunk) * kHead;
      mbar_arrive_expect_tx(&bar[i], 2u * nk * kHead * 2);
      bulk_load(smem + i * kStageBytes, k_cache + base, nk * kHead * 2, &bar[i]);
      bulk_load(smem + i * kStageBytes + kStageBytes / 2, v_cache + base, nk * kHead * 2, &bar[i]);
    }
  }
  {
    // q heads of this kv group, RoPE'd at P, this thread's 8 dims, times
    // scale * log2(e).
    float q[G][8];
    {
      const int tb = d0 & (kHalf - 1);
      const float4* cp = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(P) * kHalf + tb);
      const float4* sp = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(P) * kHalf + tb);
      const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
      const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const uint16_t* xq = qkv_new + static_cast<size_t>(s) * W + (g * G + hh) * kHead;
        const uint4 xa = __ldg(reinterpret_cast<const uint4*>(xq + tb));
        const uint4 xb = __ldg(reinterpret_cast<const uint4*>(xq + tb + kHalf));
        const float fa[8] = {bf16lo(xa.x), bf16hi(xa.x), bf16lo(xa.y), bf16hi(xa.y),
                             bf16lo(xa.z), bf16hi(xa.z), bf16lo(xa.w), bf16hi(xa.w)};
        const float fb[8] = {bf16lo(xb.x), bf16hi(xb.x), bf16lo(xb.y), bf16hi(xb.y),
                             bf16lo(xb.z), bf16hi(xb.z), bf16lo(xb.w), bf16hi(xb.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float ya, yb;
          rope_pair(fa[e], fb[e], cc[e], ss[e], ya, yb);
          q[hh][e] = (d0 < kHalf ? ya : yb) * scale_log2;
        }
      }
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them
    float m[G], l[G], o[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      m[hh] = -INFINITY;
      l[hh] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[hh][e] = 0.f;
    }
#pragma unroll 1
    for (int ci = 0; ci < n_here; ++ci) {
      const int c = c_first + ci, nk = min(kDecChunk, P + 1 - c * kDecChunk);
      uint8_t* stage = smem + ci * kStageBytes;
      const bool ok = mbar_wait(&bar[ci], 0);
      if (__syncthreads_or(!ok)) {
        // the copies did not land in time: report, give the ones in flight one
        // more bounded wait so the shared memory outlives them, leave the work
        if (tid == 0) {
          report(dev_status, ST_TIMEOUT);
          for (int i = ci; i < n_here; ++i) mbar_wait(&bar[i], 0);
        }
        return;
      }
      if (kAppend && c == n_c - 1) {
        // this chunk holds row P: write the appended k (rotated at P) and v of
        // kv head g to the caches and over the stale copy in shared memory
        const int rp = P - c * kDecChunk;
        uint16_t* ks = reinterpret_cast<uint16_t*>(stage) + rp * kHead;
        uint16_t* vs = reinterpret_cast<uint16_t*>(stage + kStageBytes / 2) + rp * kHead;
        const uint16_t* row = qkv_new + static_cast<size_t>(s) * W;
        const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
        if (tid < kHalf) {
          const uint16_t* xk = row + (heads + g) * kHead;
          const float a = __uint_as_float(static_cast<uint32_t>(xk[tid]) << 16);
          const float b = __uint_as_float(static_cast<uint32_t>(xk[tid + kHalf]) << 16);
          float ya, yb;
          rope_pair(a, b, cos_t[static_cast<size_t>(P) * kHalf + tid], sin_t[static_cast<size_t>(P) * kHalf + tid],
                    ya, yb);
          const uint32_t w2 = pack_bf16x2(ya, yb);
          const uint16_t lo = static_cast<uint16_t>(w2 & 0xffffu), hi = static_cast<uint16_t>(w2 >> 16);
          k_cache[dst + tid] = lo;
          k_cache[dst + tid + kHalf] = hi;
          ks[tid] = lo;
          ks[tid + kHalf] = hi;
        } else if (tid < kHalf + kHead) {
          const int t = tid - kHalf;
          const uint16_t v = row[(heads + kv_heads + g) * kHead + t];
          v_cache[dst + t] = v;
          vs[t] = v;
        }
        __syncthreads();
      }
      const uint16_t* Ks = reinterpret_cast<const uint16_t*>(stage);
      const uint16_t* Vs = Ks + kDecChunk * kHead;

      // scores of this thread's keys grp, grp + 16, ...
      float sc[G][kKeysPerThread];
#pragma unroll
      for (int k = 0; k < kKeysPerThread; ++k) {
        const int kk = grp + k * kGroups;
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
          sc[hh][k] = kk < nk ? v : -INFINITY;
        }
      }
      // online update of this thread's (m, l, o) with the chunk
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float mx = m[hh];
#pragma unroll
        for (int k = 0; k < kKeysPerThread; ++k) mx = fmaxf(mx, sc[hh][k]);
        const float alpha = mx == -INFINITY ? 1.f : fast_exp2(m[hh] - mx);
        m[hh] = mx;
        l[hh] *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[hh][e] *= alpha;
      }
#pragma unroll
      for (int k = 0; k < kKeysPerThread; ++k) {
        const int kk = grp + k * kGroups;
        if (kk >= nk) continue;
        const uint4 vw = *reinterpret_cast<const uint4*>(Vs + kk * kHead + d0);
        const float vf[8] = {bf16lo(vw.x), bf16hi(vw.x), bf16lo(vw.y), bf16hi(vw.y),
                             bf16lo(vw.z), bf16hi(vw.z), bf16lo(vw.w), bf16hi(vw.w)};
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float pr = fast_exp2(sc[hh][k] - m[hh]);
          l[hh] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[hh][e] = fmaf(pr, vf[e], o[hh][e]);
        }
      }
    }
    // merge the 16 key groups of this CTA: the 4 groups of a warp by
    // shuffles, then the 4 warps through shared memory
    const int wid = tid >> 5;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float mw = fmaxf(m[hh], __shfl_xor_sync(0xffffffffu, m[hh], 8));
      mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
      const float wgt = m[hh] == -INFINITY ? 0.f : fast_exp2(m[hh] - mw);
      float lw = l[hh] * wgt;
      lw += __shfl_xor_sync(0xffffffffu, lw, 8);
      lw += __shfl_xor_sync(0xffffffffu, lw, 16);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float ov = o[hh][e] * wgt;
        ov += __shfl_xor_sync(0xffffffffu, ov, 8);
        ov += __shfl_xor_sync(0xffffffffu, ov, 16);
        o[hh][e] = ov;
      }
      if ((tid & 31) < 8) {
#pragma unroll
        for (int e = 0; e < 8; ++e) red_o[(wid * G + hh) * kHead + d0 + e] = o[hh][e];
        if (lane8 == 0) {
          red_m[wid * G + hh] = mw;
          red_l[wid * G + hh] = lw;
        }
      }
    }
    __syncthreads();
    const bool single = n_parts == 1;
    float* part = partials + ((static_cast<size_t>(s) * kv_heads + g) * max_chunks + pc) * G * kPartialFloats;
    for (int e = tid; e < G * kHead; e += kDecThreads) {
      const int hh = e / kHead, d = e % kHead;
      float M = -INFINITY;
#pragma unroll
      for (int wv = 0; wv < kDecWarps; ++wv) M = fmaxf(M, red_m[wv * G + hh]);
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int wv = 0; wv < kDecWarps; ++wv) {
        const float wgt = red_m[wv * G + hh] == -INFINITY ? 0.f : fast_exp2(red_m[wv * G + hh] - M);
        Lsum = fmaf(red_l[wv * G + hh], wgt, Lsum);
        O = fmaf(red_o[(wv * G + hh) * kHead + d], wgt, O);
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
    if (!single) {
      // publish this chunk; the last CTA of (s, g) to arrive merges all chunks
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = atomicAdd(&tickets[s * kv_heads + g], 1) == n_parts - 1;
      __syncthreads();
      if (s_last) {
        __threadfence();
        // Merge in the consumed stage buffer: per-head max of m over the
        // chunks (strided over threads, then reduced), then blocks of chunk
        // weights 2^(m_c - M) in shared memory; every output sums its column
        // over the chunks with independent loads.
        const float* all = partials + (static_cast<size_t>(s) * kv_heads + g) * max_chunks * G * kPartialFloats;
        float* red = reinterpret_cast<float*>(smem);  // [G][threads], in the consumed stage 0
        float* hdr = red + G * kDecThreads;                               // [G] M, [G] L
        float* wts = hdr + 2 * G;                                         // [block][G]
        constexpr int kBlock = (kStageBytes / 4 - (kDecThreads + 2) * G) / G;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float M = -INFINITY;
          for (int cc = tid; cc < n_parts; cc += kDecThreads) M = fmaxf(M, __ldcg(all + (cc * G + hh) * kPartialFloats));
          red[hh * kDecThreads + tid] = M;
        }
        __syncthreads();
        if (tid < G) {
          float M = -INFINITY;
          for (int k = 0; k < kDecThreads; ++k) M = fmaxf(M, red[tid * kDecThreads + k]);
          hdr[tid] = M;
          hdr[G + tid] = 0.f;
        }
        float O[(G * kHead + kDecThreads - 1) / kDecThreads];
#pragma unroll
        for (int k = 0; k < (G * kHead + kDecThreads - 1) / kDecThreads; ++k) O[k] = 0.f;
        for (int c0 = 0; c0 < n_parts; c0 += kBlock) {
          const int nb = min(kBlock, n_parts - c0);
          __syncthreads();
          for (int e = tid; e < nb * G; e += kDecThreads)
            wts[e] = fast_exp2(__ldcg(all + (c0 * G + e) * kPartialFloats) - hdr[e % G]);
          __syncthreads();
          if (tid < G) {
            float Lsum = hdr[G + tid];
            for (int cc = 0; cc < nb; ++cc)
              Lsum = fmaf(__ldcg(all + ((c0 + cc) * G + tid) * kPartialFloats + 1), wts[cc * G + tid], Lsum);
            hdr[G + tid] = Lsum;
          }
#pragma unroll
          for (int k = 0; k < (G * kHead + kDecThreads - 1) / kDecThreads; ++k) {
            const int e = tid + k * kDecThreads;
            if (e < G * kHead) {
              const int hh = e / kHead, d = e % kHead;
              float acc = O[k];
#pragma unroll 8
              for (int cc = 0; cc < nb; ++cc)
                acc = fmaf(__ldcg(all + ((c0 + cc) * G + hh) * kPartialFloats + 2 + d), wts[cc * G + hh], acc);
              O[k] = acc;
            }
          }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < (G * kHead + kDecThreads - 1) / kDecThreads; ++k) {
          const int e = tid + k * kDecThreads;
          if (e < G * kHead) {
            const int hh = e / kHead, d = e % kHead;
            out[static_cast<size_t>(s) * heads * kHead + (g * G + hh) * kHead + d] = __float2bfloat16_rn(O[k] / hdr[G + hh]);
          }
        }
      }
    }
  }
}

template <int G, bool kAppend>
cudaError_t launch_decode_g(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                            float scale, const float* cos_t, const float* sin_t, int rope_len, void* k_cache,
                            void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr uint32_t smem = dec_smem_bytes<G>();
  if (dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<G, kAppend>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const int max_chunks = dec_chunks_for(cap);
  int32_t* tickets = static_cast<int32_t*>(ws);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                             align_up(static_cast<size_t>(n_seqs) * kv_heads * 4, 256));
  cudaError_t e = cudaMemsetAsync(tickets, 0, static_cast<size_t>(n_seqs) * kv_heads * 4, st);
  if (e != cudaSuccess) return e;
  dim3 grid((max_chunks + kDecPer - 1) / kDecPer, kv_heads, n_seqs);
  decode_kernel<G, kAppend><<<grid, kDecThreads, smem, st>>>(
      static_cast<const uint16_t*>(qkv_new), pos, n_seqs, heads, kv_heads, cap, scale * 1.4426950408889634f, cos_t,
      sin_t, rope_len, static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
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
                          const void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st,
                          bool append) {
  void* kc = const_cast<void*>(k_cache);
  void* vc = const_cast<void*>(v_cache);
  switch (heads / kv_heads) {
#define KIME_G(N)                                                                                                    \
  case N:                                                                                                            \
    return append ? launch_decode_g<N, true>(qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t,        \
                                             rope_len, kc, vc, out, ws, dev_status, st)                              \
                  : launch_decode_g<N, false>(qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t,       \
                                              rope_len, kc, vc, out, ws, dev_status, st);
    KIME_G(1) KIME_G(2) KIME_G(3) KIME_G(4) KIME_G(5) KIME_G(6) KIME_G(7) KIME_G(8)
#undef KIME_G
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kime
