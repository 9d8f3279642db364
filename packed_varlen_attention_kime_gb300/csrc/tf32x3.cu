// tf32x3.cu -- packed variable-length attention for FP32 qkv / FP32 out on the
// tensor cores, every product taken as three TF32 products (3xTF32).
//
// The operation is the one of the FP32 path (kime-cuda 0.0.3, src/plan.rs,
// Step::Attention, attention[f32]): RoPE at each token's position within its
// own sequence (rotate-half, float32 tables), scale, softmax over the visible
// keys, P V.  TF32 keeps 10 mantissa bits, so one TF32 product would miss the
// FP32 contract (max abs error 1e-5 against the FP64 oracle).  Each FP32
// operand x is split as x = hi + lo with hi = x rounded to TF32 (nearest, ties
// away) and lo = x - hi (exact in FP32, |lo| <= 2^-11 |x|); a product a b is
// then taken as a_lo b_hi + a_hi b_lo + a_hi b_hi on the tensor cores with FP32
// accumulation, leaving out a_lo b_lo (<= 2^-22 |a b|) and the truncation of
// lo to TF32 (<= 2^-21 |a b|): FP32-level accuracy at TF32 tensor rates.
//
// Two kernels:
//   split   one pass over the qkv rows: queries and keys rotated (the same
//           float32 evaluation as the CUDA-core FP32 kernel), queries scaled by
//           scale * log2(e) (the softmax then works in log2 units), values
//           transposed, everything split into TF32 high and low planes.  The
//           transposed values put each sequence at a column that is a multiple
//           of 4 (16 bytes), so a TMA box of a sequence's keys always starts on
//           a 16-byte boundary.
//   attend  persistent CTAs of 128 threads take (query tile, head) units from
//           the scheduler's list.  Thread r owns row r of the 128-row query
//           tile (TMEM lane r).  Key tiles are visited in 64-key halves:
//           S = Q K^T (three 128x64x64 TF32 MMA chains into TMEM), online
//           softmax in FP32 on S loaded from TMEM (exponentials on the MUFU,
//           ex2.approx: relative error about 2^-22, far inside the FP32
//           contract), P split into high and low
//           parts stored to TMEM, O += P V (three chains, A = P from TMEM,
//           B = V^T from shared memory), O rescaled in TMEM when the row max
//           moves.  Q (high, low: 64 KB) stays in shared memory for the unit;
//           the K / V^T halves (64 KB each) are double-buffered, the next one
//           loaded by TMA (as soon as the PV that read its stage is done)
//           while the current one is in the softmax.  Thread 0
//           issues the copies and the MMAs.
#include "kime_common.cuh"
#include "kime_internal.h"

namespace kime {

namespace {

constexpr int kT3Threads = 128;
constexpr int kSub = 64;                  // keys per visited half tile
constexpr uint32_t kSlabQ = kBM * 128;    // one 32-column (128-byte) slab of a 128-row tile: 16 KB
constexpr uint32_t kSlabK = kSub * 128;   // one slab of a 64-row tile: 8 KB
constexpr uint32_t kOffQh = 0, kOffQl = 2 * kSlabQ, kOffStage = 4 * kSlabQ;
constexpr uint32_t kKh = 0, kKl = 2 * kSlabK, kVh = 4 * kSlabK, kVl = 6 * kSlabK, kStageBytes = 8 * kSlabK;
constexpr uint32_t kT3Smem = kOffStage + 2 * kStageBytes + 1024;  // + slack to align the base to 1 KB
static_assert(kT3Smem <= 232448, "shared memory");
constexpr uint32_t kQBytes = 4 * kSlabQ, kKVBytes = kStageBytes;  // transaction bytes per load group
// TMEM columns: S 0..63, P high 64..127, P low 128..191, O 192..255
constexpr uint32_t kT3Cols = 256, kColPh = 64, kColPl = 128, kColO = 192;

// Instruction descriptor, kind::tf32: TF32 A and B (format 2), FP32 D, both
// K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdesc = idesc_tf32_f32(kBM, 64);  // S: 128 x 64 keys; O: 128 x 64 dims

__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(acc)
      : "memory");
}

// x rounded to TF32 (nearest, ties away from zero): the 13 low mantissa bits zero
__device__ __forceinline__ float tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// First column of sequence s in a transposed value plane (a multiple of 4;
// sequence s + 1 starts at least L_s + 1 columns later).
__host__ __device__ __forceinline__ int vt_col(int cu_s, int s) { return 4 * ((cu_s + 3) >> 2) + 4 * s; }

__device__ __forceinline__ bool visible(int i, int j, int L, int causal, int window) {
  if (j >= L) return false;
  if (causal && j > i) return false;
  if (window >= 0 && abs(i - j) > window) return false;
  return true;
}

// ------------------------------------------------------------------ split
constexpr int kSplitRows = 32;  // tokens per CTA

__global__ void __launch_bounds__(256)
    tf32_split_kernel(const float* __restrict__ qkv, const int32_t* __restrict__ cu, int n_seqs, int total,
                      int heads, int kv_heads, float qmul, const float* __restrict__ cos_t,
                      const float* __restrict__ sin_t, int rope_len, int tp, float* __restrict__ qh,
                      float* __restrict__ ql, float* __restrict__ kh, float* __restrict__ kl,
                      float* __restrict__ vh, float* __restrict__ vl) {
  __shared__ float vs[kSplitRows][kHead + 1];
  __shared__ int s_col[kSplitRows], s_pos[kSplitRows];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = blockIdx.x * kSplitRows;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  if (tid < kSplitRows) {
    const int j = j0 + tid;
    int col = -1, pos = -1;
    if (j < total) {
      // the sequence owning row j: the largest s with cu[s] <= j
      int lo = 0, hi = n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= j) lo = mid;
        else hi = mid - 1;
      }
      const int c0 = __ldg(cu + lo);
      pos = j - c0;
      // (with a malformed cu the scheduler reports it and skips the sequence;
      // here only the plane's bounds matter)
      if (pos >= 0 && c0 >= 0 && c0 <= total) {
        const long long c = static_cast<long long>(vt_col(c0, lo)) + pos;
        col = c < tp ? static_cast<int>(c) : -1;
      }
    }
    s_col[tid] = col;
    s_pos[tid] = pos;
  }
  __syncthreads();
  // queries and keys: warp w rotates tokens w, w + 8, ...; lane l takes the
  // pair (l, l + 32) of every head
  const int hq = heads * kHead, hk = kv_heads * kHead;
  for (int t = warp; t < kSplitRows; t += 8) {
    const int j = j0 + t;
    if (j >= total) break;
    const int pos = s_pos[t];
    const bool rot = pos >= 0 && pos < rope_len;  // a row of no valid sequence: not rotated
    const float c = rot ? __ldg(cos_t + static_cast<size_t>(pos) * kHalf + lane) : 1.f;
    const float s = rot ? __ldg(sin_t + static_cast<size_t>(pos) * kHalf + lane) : 0.f;
    const float* x = qkv + static_cast<size_t>(j) * W;
    for (int hd = 0; hd < heads + kv_heads; ++hd) {
      const float a = __ldg(x + hd * kHead + lane), b = __ldg(x + hd * kHead + lane + kHalf);
      float ya = a, yb = b;
      if (rot) rope_pair(a, b, c, s, ya, yb);
      float *dh, *dl;
      if (hd < heads) {
        ya *= qmul;
        yb *= qmul;
        dh = qh + static_cast<size_t>(j) * hq + hd * kHead;
        dl = ql + static_cast<size_t>(j) * hq + hd * kHead;
      } else {
        dh = kh + static_cast<size_t>(j) * hk + (hd - heads) * kHead;
        dl = kl + static_cast<size_t>(j) * hk + (hd - heads) * kHead;
      }
      const float ha = tf32_hi(ya), hb = tf32_hi(yb);
      dh[lane] = ha;
      dh[lane + kHalf] = hb;
      dl[lane] = ya - ha;
      dl[lane + kHalf] = yb - hb;
    }
  }
  // values: one kv head at a time through shared memory, written transposed
  // (consecutive threads: consecutive tokens of one dimension)
  for (int g = 0; g < kv_heads; ++g) {
    __syncthreads();
    for (int e = tid; e < kSplitRows * kHead; e += 256) {
      const int t = e / kHead, d = e % kHead, j = j0 + t;
      vs[t][d] = j < total ? __ldg(qkv + static_cast<size_t>(j) * W + (heads + kv_heads + g) * kHead + d) : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < kSplitRows * kHead; e += 256) {
      const int d = e / kSplitRows, t = e % kSplitRows;
      const int col = s_col[t];
      if (col < 0) continue;
      const float v = vs[t][d], h = tf32_hi(v);
      const size_t at = static_cast<size_t>(g * kHead + d) * tp + col;
      vh[at] = h;
      vl[at] = v - h;
    }
  }
  // runs beside the scheduler (it reads none of its output) and ends only
  // after it, so the attention kernel, which waits for this pass, also finds
  // the scheduler's lists complete
  griddep_wait();
}

// ----------------------------------------------------------------- attend
struct T3Params {
  int heads, kv_heads, window, causal;
  float* out;
  WsHeader* hdr;
  const Pair* pairs;
  int32_t* dev_status;
};

__global__ void __launch_bounds__(kT3Threads, 1)
    prefill_3xtf32_kernel(const __grid_constant__ CUtensorMap q_h, const __grid_constant__ CUtensorMap q_l,
                          const __grid_constant__ CUtensorMap k_h, const __grid_constant__ CUtensorMap k_l,
                          const __grid_constant__ CUtensorMap v_h, const __grid_constant__ CUtensorMap v_l,
                          const T3Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, kv_full[2], s_done, pv_done, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_unit;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 1 KB aligned (128-byte swizzle atoms)
  uint8_t* const sp = smem_raw + (sb - raw);

  if (tid == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&kv_full[0], 1);
    mbar_init(&kv_full[1], 1);
    mbar_init(&s_done, 1);
    mbar_init(&pv_done, 1);
    mbar_init(&drain, 1);
    fence_mbar_init();
    tma_prefetch_map(&q_h);
    tma_prefetch_map(&q_l);
    tma_prefetch_map(&k_h);
    tma_prefetch_map(&k_l);
    tma_prefetch_map(&v_h);
    tma_prefetch_map(&v_l);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, kT3Cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem, tPh = tmem + kColPh, tPl = tmem + kColPl, tO = tmem + kColO;

  griddep_wait();  // the scheduler's list and the split planes
  const int n_units = p.hdr->n_pairs * p.heads;
  const int G = p.heads / p.kv_heads;

  // barrier phases (every thread passes the same waits, so the counts agree)
  uint32_t nq = 0, ns = 0, npv = 0;
  uint32_t c = 0;                      // K/V halves consumed (all units): stage c & 1
  uint32_t issued_q = 0, issued_c = 0; // thread 0: copies started (for the wind-down)
  bool ok = true, lost = false;  // lost: thread 0's wait for the previous PV ran out

  for (;;) {
    if (tid == 0) s_unit = atomicAdd(&p.hdr->next_unit, 1);
    __syncthreads();
    const int u = s_unit;
    __syncthreads();  // every thread has read s_unit before it is rewritten
    if (u >= n_units) break;
    const Pair pr = p.pairs[u / p.heads];
    const int h = u % p.heads, g = h / G;
    const int q0 = pr.qt * kBM, q1 = min(q0 + kBM, pr.L);
    const int i = q0 + tid;
    const bool row_ok = i < pr.L;
    // the visited halves [hb, he) of the unit's key tiles
    auto half_visited = [&](int hf) {
      const int k0 = hf * kSub;
      if (k0 >= pr.L) return false;
      if (p.causal && k0 > q1 - 1) return false;
      if (p.window >= 0 && (k0 > q1 - 1 + p.window || k0 + kSub - 1 < q0 - p.window)) return false;
      return true;
    };
    int hb = 2 * pr.kt_begin, he = 2 * pr.kt_end;
    while (hb < he && !half_visited(hb)) ++hb;
    while (he > hb && !half_visited(he - 1)) --he;
    const int nsub = he - hb;
    if (nsub == 0) continue;  // (every valid row sees at least its own key)
    const int vcol = vt_col(pr.row0, pr.s);

    // copies of half number k of this unit into stage (c0 + k) & 1
    const uint32_t c0 = c;
    auto load_half = [&](int k) {
      const uint32_t cc = c0 + k, st = cc & 1;
      const int k0 = (hb + k) * kSub;
      uint8_t* base = sp + kOffStage + st * kStageBytes;
      mbar_arrive_expect_tx(&kv_full[st], kKVBytes);
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        tma_load_2d(base + kKh + a * kSlabK, &k_h, &kv_full[st], g * kHead + 32 * a, pr.row0 + k0);
        tma_load_2d(base + kKl + a * kSlabK, &k_l, &kv_full[st], g * kHead + 32 * a, pr.row0 + k0);
        tma_load_2d(base + kVh + a * kSlabK, &v_h, &kv_full[st], vcol + k0 + 32 * a, g * kHead);
        tma_load_2d(base + kVl + a * kSlabK, &v_l, &kv_full[st], vcol + k0 + 32 * a, g * kHead);
      }
      issued_c = cc + 1;
    };
    if (tid == 0) {
      // every MMA of the previous unit has completed (its last PV was waited
      // for), so Q and both stages are free
      mbar_arrive_expect_tx(&q_full, kQBytes);
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        tma_load_2d(sp + kOffQh + a * kSlabQ, &q_h, &q_full, h * kHead + 32 * a, pr.row0 + q0);
        tma_load_2d(sp + kOffQl + a * kSlabQ, &q_l, &q_full, h * kHead + 32 * a, pr.row0 + q0);
      }
      issued_q = nq + 1;
      load_half(0);
      if (nsub > 1) load_half(1);
    }
    ok = mbar_wait(&q_full, nq & 1);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    ++nq;

    float m = -INFINITY, l = 0.f;
    for (int k = 0; k < nsub; ++k, ++c) {
      const uint32_t st = c & 1;
      const int hf = hb + k, k0 = hf * kSub, kt = hf >> 1;
      const bool full = kt >= pr.full_begin && kt < pr.full_end;
      ok = mbar_wait(&kv_full[st], (c >> 1) & 1);
      ok = __syncthreads_and(ok);
      if (!ok) break;
      if (tid == 0) {
        // S = Q K^T: the two small products first, then the high one
        tc_fence_after();
        const uint32_t kb = sb + kOffStage + st * kStageBytes;
        const uint32_t A[3] = {sb + kOffQl, sb + kOffQh, sb + kOffQh};
        const uint32_t B[3] = {kb + kKh, kb + kKl, kb + kKh};
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int ks = 0; ks < kHead / 8; ++ks)
            mma_tf32_ss(tS, sdesc_sw128(A[q] + (ks >> 2) * kSlabQ + (ks & 3) * 32, 16, 1024),
                        sdesc_sw128(B[q] + (ks >> 2) * kSlabK + (ks & 3) * 32, 16, 1024), (q | ks) != 0);
        tc_commit(&s_done);
        // the next half's copies go into the stage that the previous half's
        // PV read: issued as soon as that PV is done, they have the whole
        // softmax of this half to land
        if (k > 0 && k + 1 < nsub) {
          if (mbar_wait(&pv_done, npv & 1)) load_half(k + 1);
          else lost = true;
        }
      }
      ok = mbar_wait(&s_done, ns & 1) && !lost;
      ok = __syncthreads_and(ok);
      if (!ok) break;
      ++ns;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld64_wait(tS + lane_off, sv);
      // online softmax in log2 units (q carries scale * log2(e))
      float x[64];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const bool vis = row_ok && (full || visible(i, k0 + j, pr.L, p.causal, p.window));
        x[j] = vis ? __uint_as_float(sv[j]) : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
      const float m_new = fmaxf(m, mx);
      float alpha = 1.f;
      if (m_new == -INFINITY) {
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = 0.f;
      } else {
        alpha = fast_exp2(m - m_new);
        float rs = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          x[j] = fast_exp2(x[j] - m_new);
          rs += x[j];
        }
        l = l * alpha + rs;
        m = m_new;
      }
      // PV of the previous half read P from TMEM and accumulated into O: it
      // completes before P is stored again and O is rescaled
      if (k > 0) {
        ok = mbar_wait(&pv_done, npv & 1);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        ++npv;
        tc_fence_after();
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float v = x[16 * q + e], hi = tf32_hi(v);
          ph[e] = __float_as_uint(hi);
          pl[e] = __float_as_uint(v - hi);
        }
        tmem_st16(tPh + lane_off + 16 * q, ph);
        tmem_st16(tPl + lane_off + 16 * q, pl);
      }
      if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t ov[64];
        tmem_ld64_wait(tO + lane_off, ov);
#pragma unroll
        for (int d = 0; d < kHead; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
        tmem_st64(tO + lane_off, ov);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        // O += P V: the two small products first, then the high one; the
        // unit's first half overwrites O
        tc_fence_after();
        const uint32_t vb = sb + kOffStage + st * kStageBytes;
        const uint32_t A[3] = {tPl, tPh, tPh};
        const uint32_t B[3] = {vb + kVh, vb + kVl, vb + kVh};
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int ks = 0; ks < kSub / 8; ++ks)
            mma_tf32_ts(tO, A[q] + ks * 8, sdesc_sw128(B[q] + (ks >> 2) * kSlabK + (ks & 3) * 32, 16, 1024),
                        (k | q | ks) != 0);
        tc_commit(&pv_done);
      }
    }
    if (!ok) break;
    // epilogue: the last PV, then O / l
    ok = mbar_wait(&pv_done, npv & 1);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    ++npv;
    tc_fence_after();
    uint32_t ov[64];
    tmem_ld64_wait(tO + lane_off, ov);
    tc_fence_before();
    if (row_ok) {
      const float inv = 1.f / l;
      float* dst = p.out + static_cast<size_t>(pr.row0 + i) * p.heads * kHead + h * kHead;
#pragma unroll
      for (int d = 0; d < kHead; d += 4)
        *reinterpret_cast<float4*>(dst + d) =
            make_float4(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv,
                        __uint_as_float(ov[d + 2]) * inv, __uint_as_float(ov[d + 3]) * inv);
    }
    __syncthreads();  // every O load is done before the next unit's first PV
  }

  if (!ok) {
    // a wait ran past its limit: report, then let the copies and MMAs this
    // CTA started finish (bounded) before TMEM is freed
    if (tid == 0) {
      report(p.dev_status, ST_TIMEOUT);
      if (issued_q > nq) mbar_wait(&q_full, nq & 1);
      for (uint32_t cc = c; cc < issued_c; ++cc) mbar_wait(&kv_full[cc & 1], (cc >> 1) & 1);
      tc_commit(&drain);
      mbar_wait(&drain, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kT3Cols);
  }
}

}  // namespace

cudaError_t launch_tf32_clear(int n_seqs, int total, int heads, int kv_heads, void* ws, cudaStream_t st) {
  // the gaps between the sequences' value columns read as zeros (a key tile
  // of a sequence may reach into them; its P there is 0, and 0 * 0 = 0)
  const Tf32Planes pl = tf32_planes(n_seqs, total, heads, kv_heads);
  return cudaMemsetAsync(static_cast<char*>(ws) + pl.vh, 0, pl.end - pl.vh, st);
}

cudaError_t launch_tf32_split(const float* qkv, const int32_t* cu, int n_seqs, int total, int heads, int kv_heads,
                              float scale, const float* cos_t, const float* sin_t, int rope_len, void* ws,
                              cudaStream_t st) {
  const Tf32Planes pl = tf32_planes(n_seqs, total, heads, kv_heads);
  char* w = static_cast<char*>(ws);
  // launched with programmatic stream serialization: it starts while the
  // scheduler (which lets dependents start at once) still runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((total + kSplitRows - 1) / kSplitRows);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tf32_split_kernel, qkv, cu, n_seqs, total, heads, kv_heads,
                            scale * 1.4426950408889634f, cos_t, sin_t, rope_len, pl.tp,
                            reinterpret_cast<float*>(w + pl.qh), reinterpret_cast<float*>(w + pl.ql),
                            reinterpret_cast<float*>(w + pl.kh), reinterpret_cast<float*>(w + pl.kl),
                            reinterpret_cast<float*>(w + pl.vh), reinterpret_cast<float*>(w + pl.vl));
}

cudaError_t launch_prefill_3xtf32(const CUtensorMap* q_h, const CUtensorMap* q_l, const CUtensorMap* k_h,
                                  const CUtensorMap* k_l, const CUtensorMap* v_h, const CUtensorMap* v_l,
                                  int heads, int kv_heads, int window, int causal, float* out, void* ws,
                                  int32_t* dev_status, cudaStream_t st) {
  static int configured[64] = {0};
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_3xtf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kT3Smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  T3Params prm;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.window = window;
  prm.causal = causal;
  prm.out = out;
  prm.hdr = static_cast<WsHeader*>(ws);
  prm.pairs = ws_pairs(ws);
  prm.dev_status = dev_status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kT3Threads);
  cfg.dynamicSmemBytes = kT3Smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_3xtf32_kernel, *q_h, *q_l, *k_h, *k_l, *v_h, *v_l, prm);
}

}  // namespace kime
