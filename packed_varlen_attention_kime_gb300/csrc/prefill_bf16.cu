// prefill_bf16.cu -- packed variable-length attention over a BF16 fused qkv
// buffer on the sm_103a tensor cores (tcgen05, TMEM accumulators, TMA).
//
// What it computes (per sequence s, head h, local query i of a length-L
// sequence): softmax over the visible keys j of scale * <rope(q_i, i),
// rope(k_j, j)>, times v_j, where q is head h of the row, k/v are kv head
// h / (heads/kv_heads) (ffai-argus 0.7.3 src/text.rs, TextTower::block GQA
// fold), RoPE is rotate-half with the cos/sin tables of kime-cuda 0.0.3
// src/plan.rs (fn rope_tables), positions restart at every sequence
// (kime-cpu 0.0.17 src/kime_cpu/plan.rs, Step::Rope), and key j is visible
// when j <= i if causal and |i - j| <= window if window >= 0 (kime-cuda
// Op::Attention: window None = -1).  Masked keys are skipped, never written
// as -inf (ffai-argus src/text.rs module doc and CausalSoftmax).
//
// Structure: persistent CTAs of 128 threads take (pair, head) units from the
// device schedule.  Per unit:
//   TMA  Q tile [128 rows x 64] (128-byte swizzle) -> RoPE in shared memory
//   per visited key tile (double-buffered TMA of K and V):
//     RoPE on K in shared memory, fence.proxy.async
//     tcgen05.mma  S[TMEM 128x128 f32] = Q . K^T         (4 x K=16)
//     tcgen05.ld S, online softmax in registers (base-2, masked keys skipped)
//     P (bf16) -> shared memory, swizzled K-major
//     tcgen05.mma  PV[TMEM 128x64 f32] = P . V           (8 x K=16, V MN-major)
//     tcgen05.ld PV, O = O*alpha + PV in registers
//   epilogue: O / l -> bf16 rows that belong to the sequence.
// Thread t owns query row t of the tile = TMEM lane t.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kTileBytes = kBM * kHead * 2;  // 16 KB: 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;      // 2 stages
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes;  // 2 stages
constexpr uint32_t kOffP = kOffV + 2 * kTileBytes;  // 2 halves (keys 0..63, 64..127)
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 128 + 1024;  // + barriers + alignment slack
constexpr uint32_t kTmemCols = 256;                     // S: 0..127, PV: 128..191
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, 0, 1);

struct Bars {
  uint64_t q, kv[2], mma;
  uint32_t tmem_base;
  int unit;
};

// RoPE (rotate-half) of row r of a 128-byte-swizzled [128 x 64] bf16 tile, in
// place, at table row (c, s).  16-byte chunk k of row r sits at chunk k ^ (r & 7).
__device__ __forceinline__ void rope_row_sw128(uint8_t* tile, int r, const float* __restrict__ c,
                                               const float* __restrict__ s) {
  uint8_t* row = tile + r * 128;
  const int sw = r & 7;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4* plo = reinterpret_cast<uint4*>(row + ((k ^ sw) << 4));
    uint4* phi = reinterpret_cast<uint4*>(row + (((k + 4) ^ sw) << 4));
    const uint4 a = *plo, b = *phi;
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(c + 8 * k));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(c + 8 * k + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(s + 8 * k));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(s + 8 * k + 4));
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a0, a1, b0, b1;
      rope_pair(bf16lo(aw[e]), bf16lo(bw[e]), cc[2 * e], ss[2 * e], a0, b0);
      rope_pair(bf16hi(aw[e]), bf16hi(bw[e]), cc[2 * e + 1], ss[2 * e + 1], a1, b1);
      ya[e] = pack_bf16x2(a0, a1);
      yb[e] = pack_bf16x2(b0, b1);
    }
    *plo = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *phi = make_uint4(yb[0], yb[1], yb[2], yb[3]);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap qkv_map, int heads, int kv_heads, int window,
                        int causal, float scale_log2, const float* __restrict__ cos_t,
                        const float* __restrict__ sin_t, __nv_bfloat16* __restrict__ out, WsHeader* hdr,
                        const Pair* __restrict__ pairs, int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sP = smem + kOffP;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = heads / kv_heads;
  const int n_units = hdr->n_pairs * heads;

  if (tid == 0) {
    tma_prefetch_map(&qkv_map);
    mbar_init(&bars->q, 1);
    mbar_init(&bars->kv[0], 1);
    mbar_init(&bars->kv[1], 1);
    mbar_init(&bars->mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_S = tmem;
  const uint32_t tmem_PV = tmem + 128;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  uint32_t ph_q = 0, ph_kv[2] = {0, 0}, ph_mma = 0;
  bool failed = false;
  // Thread 0 tracks copies / MMAs it issued that nobody has waited for yet.
  int pend_q = 0, pend_kv[2] = {0, 0}, pend_mma = 0;

  auto wait = [&](uint64_t* bar, uint32_t& ph) {
    if (!failed && !mbar_wait(bar, ph)) failed = true;
    ph ^= 1;
  };

  for (;;) {
    if (tid == 0) bars->unit = atomicAdd(&hdr->next_unit, 1);
    __syncthreads();
    const int u = bars->unit;
    if (u >= n_units) break;
    const Pair pr = pairs[u / heads];
    const int h = u % heads, g = h / G;
    const int q0 = pr.qt * kBM;
    const int i = q0 + tid;  // this thread's query row (local)
    const bool row_ok = i < pr.L;
    const int kx = (heads + g) * kHead, vx = (heads + kv_heads + g) * kHead;

    if (tid == 0) {
      mbar_arrive_expect_tx(&bars->q, kTileBytes);
      tma_load_2d(sQ, &qkv_map, &bars->q, h * kHead, pr.row0 + q0);
      pend_q = 1;
      mbar_arrive_expect_tx(&bars->kv[0], 2 * kTileBytes);
      tma_load_2d(sK, &qkv_map, &bars->kv[0], kx, pr.row0 + pr.kt_begin * kBN);
      tma_load_2d(sV, &qkv_map, &bars->kv[0], vx, pr.row0 + pr.kt_begin * kBN);
      pend_kv[0] = 1;
    }
    wait(&bars->q, ph_q);
    if (tid == 0) pend_q = 0;
    if (row_ok) rope_row_sw128(sQ, tid, cos_t + static_cast<size_t>(i) * kHalf, sin_t + static_cast<size_t>(i) * kHalf);
    fence_proxy_async_smem();

    float o[kHead];
#pragma unroll
    for (int d = 0; d < kHead; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int kt = pr.kt_begin; kt < pr.kt_end; ++kt) {
      const int st = (kt - pr.kt_begin) & 1;
      const int k0 = kt * kBN;
      uint8_t* sKs = sK + st * kTileBytes;
      uint8_t* sVs = sV + st * kTileBytes;
      if (tid == 0 && kt + 1 < pr.kt_end) {  // prefetch the next key tile into the other stage
        mbar_arrive_expect_tx(&bars->kv[st ^ 1], 2 * kTileBytes);
        tma_load_2d(sK + (st ^ 1) * kTileBytes, &qkv_map, &bars->kv[st ^ 1], kx, pr.row0 + k0 + kBN);
        tma_load_2d(sV + (st ^ 1) * kTileBytes, &qkv_map, &bars->kv[st ^ 1], vx, pr.row0 + k0 + kBN);
        pend_kv[st ^ 1] = 1;
      }
      wait(&bars->kv[st], ph_kv[st]);
      if (tid == 0) pend_kv[st] = 0;
      if (k0 + tid < pr.L)
        rope_row_sw128(sKs, tid, cos_t + static_cast<size_t>(k0 + tid) * kHalf,
                       sin_t + static_cast<size_t>(k0 + tid) * kHalf);
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(failed)) { failed = true; break; }

      // S = Q . K^T
      if (tid == 0) {
        tc_fence_after();
        const uint32_t aq = smem_u32(sQ), bk = smem_u32(sKs);
#pragma unroll
        for (int ks = 0; ks < kHead / 16; ++ks)
          tc_mma_ss(tmem_S, sdesc_sw128(aq + ks * 32, 16, 1024), sdesc_sw128(bk + ks * 32, 16, 1024), kIdescS,
                    ks > 0);
        tc_commit(&bars->mma);
        pend_mma = 1;
      }
      wait(&bars->mma, ph_mma);
      if (tid == 0) pend_mma = 0;
      tc_fence_after();

      // Online softmax over this tile's 128 keys, in two passes over the S
      // columns in TMEM (row max, then exponentials), 32 columns at a time.
      const bool full = kt >= pr.full_begin && kt < pr.full_end;
      auto logit = [&](int j, uint32_t raw) -> float {
        const float x = __uint_as_float(raw) * scale_log2;
        if (!row_ok) return -INFINITY;
        if (full) return x;
        const int jj = k0 + j;
        bool vis = jj < pr.L;
        if (causal) vis = vis && jj <= i;
        if (window >= 0) vis = vis && abs(i - jj) <= window;
        return vis ? x : -INFINITY;
      };
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tmem_S + lane_off + c * 32, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, logit(c * 32 + e, r[e]));
      }
      const float m_new = fmaxf(m, mx);
      // A row with every key so far masked keeps m = -inf; its P is all zero.
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m - m_use);
      float rowsum = 0.f;
      // P row -> shared memory: keys 0..63 in half 0, 64..127 in half 1, each a
      // 128-byte-swizzled K-major tile.
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tmem_S + lane_off + c * 32, r);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint32_t pw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = c * 32 + q8 * 8 + 2 * e;
            const float p0 = fast_exp2(logit(j, r[q8 * 8 + 2 * e]) - m_use);
            const float p1 = fast_exp2(logit(j + 1, r[q8 * 8 + 2 * e + 1]) - m_use);
            rowsum += p0 + p1;
            pw[e] = pack_bf16x2(p0, p1);
          }
          const int cc = c * 4 + q8;  // 16-byte chunk of the P row
          uint8_t* dst = sP + (cc >> 3) * kTileBytes + tid * 128 + (((cc & 7) ^ (tid & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
      }
      m = m_new;
      l = l * alpha + rowsum;
#pragma unroll
      for (int d = 0; d < kHead; ++d) o[d] *= alpha;
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(failed)) { failed = true; break; }

      // PV = P . V
      if (tid == 0) {
        tc_fence_after();
        const uint32_t ap = smem_u32(sP), bv = smem_u32(sVs);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          tc_mma_ss(tmem_PV, sdesc_sw128(ap + (ks >> 2) * kTileBytes + (ks & 3) * 32, 16, 1024),
                    sdesc_sw128(bv + ks * 2048, 0, 1024), kIdescPV, ks > 0);
        tc_commit(&bars->mma);
        pend_mma = 1;
      }
      wait(&bars->mma, ph_mma);
      if (tid == 0) pend_mma = 0;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kHead / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tmem_PV + lane_off + c * 32, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[c * 32 + e] += __uint_as_float(r[e]);
      }
      tc_fence_before();
      if (__syncthreads_or(failed)) { failed = true; break; }
    }
    if (failed) break;

    if (row_ok) {
      const float inv = 1.f / l;
      __nv_bfloat16* dst = out + static_cast<size_t>(pr.row0 + i) * heads * kHead + h * kHead;
#pragma unroll
      for (int d = 0; d < kHead; d += 8) {
        uint4 w;
        w.x = pack_bf16x2(o[d] * inv, o[d + 1] * inv);
        w.y = pack_bf16x2(o[d + 2] * inv, o[d + 3] * inv);
        w.z = pack_bf16x2(o[d + 4] * inv, o[d + 5] * inv);
        w.w = pack_bf16x2(o[d + 6] * inv, o[d + 7] * inv);
        *reinterpret_cast<uint4*>(dst + d) = w;
      }
    }
    __syncthreads();  // bars->unit is rewritten at the top
  }

  if (failed) {
    // Wind down after a timed-out wait: give copies and MMAs still in flight a
    // bounded chance to land before the shared memory and TMEM go away.
    if (tid == 0) {
      report(dev_status, ST_TIMEOUT);
      if (pend_q) mbar_wait(&bars->q, ph_q);
      if (pend_kv[0]) mbar_wait(&bars->kv[0], ph_kv[0]);
      if (pend_kv[1]) mbar_wait(&bars->kv[1], ph_kv[1]);
      if (pend_mma) mbar_wait(&bars->mma, ph_mma);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill_bf16(const CUtensorMap* qkv_map, const int32_t* cu, int n_seqs, int total, int heads,
                                int kv_heads, int window, int causal, float scale, const float* cos_t,
                                const float* sin_t, void* out, void* ws, int max_pairs, int32_t* dev_status,
                                cudaStream_t st) {
  (void)cu; (void)n_seqs; (void)total; (void)max_pairs;
  static int configured[64] = {0};
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  const Pair* pairs = reinterpret_cast<const Pair*>(static_cast<char*>(ws) + sizeof(WsHeader));
  const float scale_log2 = scale * 1.4426950408889634f;
  prefill_bf16_kernel<<<sms, kThreads, kSmemBytes, st>>>(*qkv_map, heads, kv_heads, window, causal, scale_log2,
                                                          cos_t, sin_t, static_cast<__nv_bfloat16*>(out), hdr,
                                                          pairs, dev_status);
  return cudaGetLastError();
}

}  // namespace kime
