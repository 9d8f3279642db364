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
// One kernel, after the scheduler: persistent CTAs of 512 threads over
// (128-row query tile, head) units of the scheduler's list, reading the FP32
// qkv rows as they are and visiting the unit's keys in 64-key halves:
//     warps 0-7   softmax: warps w and w + 4 share TMEM lanes 32 (w mod 4) ..
//                 +31 (rows of the tile) and take key columns 0-31 and 32-63
//                 of each half; they exchange their partial row maxima
//                 through shared memory.  FP32 online softmax (exponentials on
//                 the MUFU, ex2.approx: relative error about 2^-22), P split
//                 into TF32 high and low parts stored to TMEM, O / l at the
//                 end.  At the start of a unit the same warps read its raw
//                 query tile from shared memory, rotate it, multiply it by
//                 scale * log2(e) (the softmax then works in base 2) and store
//                 its high and low parts in TMEM: the A operand of S = Q K^T.
//     warps 8-11  operand preparation: each half's keys, as loaded, rotated
//                 at their positions (the float32 evaluation of every kernel
//                 here) and split in place (high parts over the raw values,
//                 low parts beside them); its values split and transposed
//                 (V^T is the K-major B operand of O += P V; the TF32 MMA
//                 takes its operands K-major here)
//     warp 12     TMA producer of the raw query tiles and the key halves (a
//                 3-stage ring); it also claims the units
//     warp 13     TMA producer of the value halves (a 2-stage ring)
//     warps 14-15 MMA issuers (one thread each; one thread issuing alone
//                 cannot keep up with these small MMAs): warp 14 issues S(h) =
//                 Q K^T as three 128x64x64 TF32 chains, A from TMEM; warp 15
//                 O += P(h) V(h) as three chains, A = P from TMEM.  With three
//                 S buffers S(h+1) runs while the softmax works on S(h) and
//                 PV(h) while it works on S(h+1).  The next unit's queries
//                 are stored to TMEM before the epilogue of the current one,
//                 so S of its first half runs while the current unit's last
//                 PV does.
// The softmax moves its reference maximum lazily (only when a row's maximum
// exceeds it by more than 2^8; P then stays below 2^8 and O is rescaled in
// TMEM), so it almost never touches O before the epilogue.
//
// TMEM (512 columns): S 0..191 (three buffers of 64; the softmax writes P's
// high parts over the S it has read), P low 192..319 (two buffers), O
// 320..383, Q high 384..447, Q low 448..511.  Per S buffer a barrier says
// when the PV that read its P has completed: the S issuer waits for it
// before reusing the buffer (so it can run two halves ahead of the PVs), and
// the softmax waits for it only to reuse a P-low buffer or to rescale O.
// Every wait is bounded in time; on a timeout every role winds down.
#include "kime_common.cuh"
#include "kime_internal.h"

namespace kime {

namespace {

constexpr int kT3Threads = 512;
constexpr int kSub = 64;                 // keys per visited half tile
constexpr int kKStages = 3, kVStages = 2;
constexpr uint32_t kSlabQ = kBM * 128;   // one 32-column (128-byte) slab of a 128-row tile: 16 KB
constexpr uint32_t kSlabK = kSub * 128;  // one slab of a 64-row tile: 8 KB
// shared memory, offsets from a 1 KB aligned base: the raw query tile, the
// key stages and the V^T stages (high parts, where the loads land, then low
// parts; two slabs each)
constexpr uint32_t kHalfBytes = 2 * kSlabK;  // one operand of one half: 16 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 2 * kSlabQ;
constexpr uint32_t kOffV = kOffK + kKStages * 2 * kHalfBytes;
constexpr uint32_t kT3Smem = kOffV + kVStages * 2 * kHalfBytes + 1024;  // + slack to align the base to 1 KB
static_assert(kT3Smem + 4096 <= 232448, "shared memory (dynamic + the barrier block)");
constexpr uint32_t kColS = 0, kColPl = 192, kColO = 320, kColQh = 384, kColQl = 448;
constexpr int kSBufs = 3;  // S / P-high buffers
constexpr uint32_t kT3Cols = 512;
constexpr float kLazy = 8.f;       // the reference max moves when exceeded by more (log2 units)

// Instruction descriptor, kind::tf32: TF32 A and B (format 2), FP32 D, both
// K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdesc = idesc_tf32_f32(kBM, 64);  // S: 128 x 64 keys; O: 128 x 64 dims

// D[tmem] (+)= A[tmem] B[smem], kind::tf32
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

__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Keys of one half, in place: the raw tile (two slabs: dims 0-31 and 32-63,
// 64 rows, 128-byte swizzle) rotated at positions k0 + j (rows at or past L
// are masked keys: left unrotated, their table rows may not exist) and split,
// high parts over the raw values, low parts into kl at the same offsets.
// Element (j, d) and its rotation partner (j, d + 32) sit at the same offset
// of the two slabs; the 16-byte chunk at offset o of a slab holds row o / 128,
// dims 4c .. 4c + 3 with c = (o / 16 mod 8) xor (row mod 8).  The 128
// threads of the split warps take consecutive chunks.
__device__ __forceinline__ void prep_keys(uint8_t* kh, uint8_t* kl, int k0, int L, const float* __restrict__ cos_t,
                                          const float* __restrict__ sin_t, int ct) {
  // every load first (the table rows come from L2), then the arithmetic and the stores
  float4 a[4], b[4], cs[4], sn[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int cp = ct + 128 * it;
    const int j = cp >> 3, c = (cp & 7) ^ (j & 7);
    a[it] = *reinterpret_cast<const float4*>(kh + cp * 16);
    b[it] = *reinterpret_cast<const float4*>(kh + kSlabK + cp * 16);
    const int pos = min(k0 + j, L - 1);  // (rows at or past L are not rotated below)
    cs[it] = __ldg(reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(pos) * kHalf + 4 * c));
    sn[it] = __ldg(reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(pos) * kHalf + 4 * c));
  }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int cp = ct + 128 * it;
    float4 x = a[it], y = b[it];
    if (k0 + (cp >> 3) < L) {
      rope_pair(a[it].x, b[it].x, cs[it].x, sn[it].x, x.x, y.x);
      rope_pair(a[it].y, b[it].y, cs[it].y, sn[it].y, x.y, y.y);
      rope_pair(a[it].z, b[it].z, cs[it].z, sn[it].z, x.z, y.z);
      rope_pair(a[it].w, b[it].w, cs[it].w, sn[it].w, x.w, y.w);
    }
    const float4 hx = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
    const float4 hy = make_float4(tf32_hi(y.x), tf32_hi(y.y), tf32_hi(y.z), tf32_hi(y.w));
    *reinterpret_cast<float4*>(kh + cp * 16) = hx;
    *reinterpret_cast<float4*>(kh + kSlabK + cp * 16) = hy;
    *reinterpret_cast<float4*>(kl + cp * 16) = make_float4(x.x - hx.x, x.y - hx.y, x.z - hx.z, x.w - hx.w);
    *reinterpret_cast<float4*>(kl + kSlabK + cp * 16) = make_float4(y.x - hy.x, y.y - hy.y, y.z - hy.z, y.w - hy.w);
  }
}

// ----------------------------------------------------------------- attend
// A unit as the producer publishes it: query tile q0 .. q0 + 127 of sequence
// s (rows row0 .. row0 + L - 1), head h (kv head g); halves [hb, hb + nsub)
// of 64 keys, of which [ffb, ffe) are seen whole by every row of the tile.
// u < 0 ends the list.
struct UnitInfo {
  int32_t u, s, h, g, row0, L, q0, hb, nsub, ffb, ffe;
};

struct Shared {
  uint64_t unit_full[2], unit_empty[2];
  uint64_t q_raw_full, q_raw_empty;  // the raw query tile in shared memory
  uint64_t q_ready;                  // Q high / low stored in TMEM (one arrival per softmax warp)
  uint64_t q_free;                   // every S of a unit has completed (its Q columns may be rewritten)
  uint64_t k_raw_full[kKStages], k_ready[kKStages], k_empty[kKStages];  // loaded, split (one arrival per key split warp), read by S
  uint64_t v_raw_full[kVStages], v_ready[kVStages], v_empty[kVStages];  // the same for V^T, read by PV
  uint64_t s_full[kSBufs];  // S(h) computed, by S buffer h mod 3
  uint64_t p_full[kSBufs];  // P(h) stored, O rescaled (one arrival per softmax warp)
  uint64_t pv_buf[kSBufs];  // PV(h) has completed
  uint64_t o_free;     // the epilogue has read O (one arrival per softmax warp)
  uint64_t drain[2];  // wind-down after an abort: each issuer's last commit
  UnitInfo info[2];
  float xch[2][2][kBM];  // partial row maxima: [buffer][column half][row]
  float xl[2][kBM];      // partial row sums at the epilogue: [column half][row]
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Shared) <= 4096, "barrier block");

struct T3Params {
  int heads, kv_heads, window, causal;
  float qmul;  // scale * log2(e)
  const float* cos_t;
  const float* sin_t;
  float* out;
  WsHeader* hdr;
  const Pair* pairs;
  int32_t* dev_status;
};

// kNarrow: a window of at most 64; every 64-key half is then partial for some
// row of the tile, so every half takes the partial path (the full-half code
// would only take room).  Same bits.
template <bool kNarrow>
__global__ void __launch_bounds__(kT3Threads, 1)
    prefill_3xtf32_kernel(const __grid_constant__ CUtensorMap qkv_map, const T3Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared shs;
  Shared* sh = &shs;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_map(&qkv_map);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->unit_full[i], 1);
      mbar_init(&sh->unit_empty[i], 8);  // softmax, 4 split warps, V producer, both issuers
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&sh->s_full[i], 1);
      mbar_init(&sh->p_full[i], 8);
      mbar_init(&sh->pv_buf[i], 1);
    }
    mbar_init(&sh->q_raw_full, 1);
    mbar_init(&sh->q_raw_empty, 8);
    mbar_init(&sh->q_ready, 8);
    mbar_init(&sh->q_free, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&sh->k_raw_full[i], 1);
      mbar_init(&sh->k_ready[i], 4);
      mbar_init(&sh->k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&sh->v_raw_full[i], 1);
      mbar_init(&sh->v_ready[i], 4);
      mbar_init(&sh->v_empty[i], 1);
    }

    mbar_init(&sh->o_free, 8);
    mbar_init(&sh->drain[0], 1);
    mbar_init(&sh->drain[1], 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh->tmem_base, kT3Cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  volatile int32_t* abort_flag = &sh->abort;

  // Bounded wait; a timeout anywhere raises the CTA's abort flag, after which
  // every wait that would block returns false at once and every role leaves
  // its loop.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(p.dev_status, ST_TIMEOUT);
    return false;
  };

  if (warp == 12) {
    if (lane == 0) {
      // ------------------------------------------- TMA producer: units, Q, keys
      griddep_wait();  // the scheduler's list
      const int n_units = p.hdr->n_pairs * p.heads;
      const int G = p.heads / p.kv_heads;
      uint32_t n = 0, nq = 0, c = 0;  // units published, query tiles and key halves loaded
      bool ok = true;
      for (;; ++n) {
        const int slot = n & 1;
        if (!(ok = wait(&sh->unit_empty[slot], ((n >> 1) & 1) ^ 1))) break;
        UnitInfo inf;
        inf.u = -1;
        for (;;) {
          const int u = atomicAdd(&p.hdr->next_unit, 1);
          if (u >= n_units) break;
          const Pair pr = p.pairs[u / p.heads];
          const int q0 = pr.qt * kBM, q1 = min(q0 + kBM, pr.L);
          // the halves of the pair's key tiles that hold a visible key
          auto visited = [&](int hf) {
            const int k0 = hf * kSub;
            if (k0 >= pr.L) return false;
            if (p.causal && k0 > q1 - 1) return false;
            if (p.window >= 0 && (k0 > q1 - 1 + p.window || k0 + kSub - 1 < q0 - p.window)) return false;
            return true;
          };
          int hb = 2 * pr.kt_begin, he = 2 * pr.kt_end;
          while (hb < he && !visited(hb)) ++hb;
          while (he > hb && !visited(he - 1)) --he;
          if (he == hb) continue;  // (every valid row sees at least its own key)
          inf.u = u;
          inf.s = pr.s;
          inf.h = u % p.heads;
          inf.g = inf.h / G;
          inf.row0 = pr.row0;
          inf.L = pr.L;
          inf.q0 = q0;
          inf.hb = hb;
          inf.nsub = he - hb;
          inf.ffb = 2 * pr.full_begin;
          inf.ffe = 2 * pr.full_end;
          break;
        }
        sh->info[slot] = inf;
        mbar_arrive(&sh->unit_full[slot]);
        if (inf.u < 0) break;
        // the raw query tile: two slabs of 32 dims, each as two 64-row boxes
        if (!(ok = wait(&sh->q_raw_empty, (nq & 1) ^ 1))) break;
        mbar_arrive_expect_tx(&sh->q_raw_full, 2 * kSlabQ);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int b = 0; b < 2; ++b)
            tma_load_2d(smem + kOffQ + a * kSlabQ + b * kSlabK, &qkv_map, &sh->q_raw_full, inf.h * kHead + 32 * a,
                        inf.row0 + inf.q0 + 64 * b);
        ++nq;
        for (int k = 0; k < inf.nsub; ++k, ++c) {
          const uint32_t st = c % kKStages;
          if (!(ok = wait(&sh->k_empty[st], ((c / kKStages) & 1) ^ 1))) break;
          uint8_t* kb = smem + kOffK + st * 2 * kHalfBytes;  // the raw keys land in the high part
          mbar_arrive_expect_tx(&sh->k_raw_full[st], kHalfBytes);
#pragma unroll
          for (int a = 0; a < 2; ++a)
            tma_load_2d(kb + a * kSlabK, &qkv_map, &sh->k_raw_full[st], (p.heads + inf.g) * kHead + 32 * a,
                        inf.row0 + (inf.hb + k) * kSub);
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // every copy this thread issued lands before the CTA releases its
        // shared memory: the last fill of each stage, the last query tile
        for (uint32_t st = 0; st < kKStages; ++st)
          if (c > st) mbar_wait(&sh->k_raw_full[st], (((c - 1) - ((c - 1 - st) % kKStages)) / kKStages) & 1);
        if (nq > 0) mbar_wait(&sh->q_raw_full, (nq - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    if (lane == 0) {
      // -------------------------------------------------- TMA producer: V^T
      uint32_t n = 0, c = 0;
      bool ok = true;
      for (;; ++n) {
        const int slot = n & 1;
        if (!(ok = wait(&sh->unit_full[slot], (n >> 1) & 1))) break;
        const UnitInfo inf = sh->info[slot];
        mbar_arrive(&sh->unit_empty[slot]);
        if (inf.u < 0) break;
        const int vx = (p.heads + p.kv_heads + inf.g) * kHead;
        for (int k = 0; k < inf.nsub; ++k, ++c) {
          const uint32_t st = c % kVStages;
          if (!(ok = wait(&sh->v_empty[st], ((c / kVStages) & 1) ^ 1))) break;
          uint8_t* vl = smem + kOffV + st * 2 * kHalfBytes + kHalfBytes;  // the raw values land in the low part
          mbar_arrive_expect_tx(&sh->v_raw_full[st], kHalfBytes);
#pragma unroll
          for (int a = 0; a < 2; ++a)
            tma_load_2d(vl + a * kSlabK, &qkv_map, &sh->v_raw_full[st], vx + 32 * a, inf.row0 + (inf.hb + k) * kSub);
        }
        if (!ok) break;
      }
      if (*abort_flag)
        for (uint32_t st = 0; st < kVStages; ++st)
          if (c > st) mbar_wait(&sh->v_raw_full[st], (((c - 1) - ((c - 1 - st) % kVStages)) / kVStages) & 1);
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------ operand preparation
    // The four warps pass the same named barriers (id 6, 128 threads): one
    // per unit, one per half; a failed wait is carried to the next of them.
    const int ct = tid - 256, cw = warp - 8;  // 0 .. 127, 0 .. 3
    uint32_t n = 0, h = 0;
    bool ok = true;
    for (;; ++n) {
      const int slot = n & 1;
      ok = __all_sync(0xffffffffu, ok && wait(&sh->unit_full[slot], (n >> 1) & 1));
      if (named_bar_or(6, 128, !ok)) break;
      const UnitInfo inf = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->unit_empty[slot]);
      if (inf.u < 0) break;
      for (int k = 0; k < inf.nsub; ++k, ++h) {
        const uint32_t ks = h % kKStages, vs = h % kVStages;
        // keys: rotated at their positions and split in place
        ok = __all_sync(0xffffffffu, ok && wait(&sh->k_raw_full[ks], (h / kKStages) & 1));
        if (ok) {
          uint8_t* kb = smem + kOffK + ks * 2 * kHalfBytes;
          prep_keys(kb, kb + kHalfBytes, (inf.hb + k) * kSub, inf.L, p.cos_t, p.sin_t, ct);
          fence_proxy_async_smem();  // visible to the tensor core
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->k_ready[ks]);
        }
        // values: the raw tile (slabs of 32 dims, 64 key rows, in the low
        // part) read as 4x4 blocks, then written transposed (slabs of 32
        // keys, 64 dim rows): high parts into the high part, low parts over
        // the raw tile.  Lane (kg_lo, dg_lo) = (lane & 7, lane >> 3) takes
        // blocks of keys 4 kg .. 4 kg + 3 and dims 4 dg .. 4 dg + 3; every
        // 16-byte access of a warp spreads over all eight chunk positions.
        ok = __all_sync(0xffffffffu, ok && wait(&sh->v_raw_full[vs], (h / kVStages) & 1));
        uint8_t* vh = smem + kOffV + vs * 2 * kHalfBytes;
        uint8_t* vl = vh + kHalfBytes;
        float4 blk[2][4];
        if (ok) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 2 * cw + i, kg = (lane & 7) + 8 * (c & 1), dg = (lane >> 3) + 4 * (c >> 1);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 4 * kg + e;
              blk[i][e] = *reinterpret_cast<const float4*>(vl + (dg >> 3) * kSlabK + j * 128 +
                                                           (((dg & 7) ^ (j & 7)) << 4));
            }
          }
        }
        // every raw value has been read before any low part overwrites it
        if (named_bar_or(6, 128, !ok)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = 2 * cw + i, kg = (lane & 7) + 8 * (c & 1), dg = (lane >> 3) + 4 * (c >> 1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 4 * dg + e;
            const float4 v = e == 0 ? make_float4(blk[i][0].x, blk[i][1].x, blk[i][2].x, blk[i][3].x)
                           : e == 1 ? make_float4(blk[i][0].y, blk[i][1].y, blk[i][2].y, blk[i][3].y)
                           : e == 2 ? make_float4(blk[i][0].z, blk[i][1].z, blk[i][2].z, blk[i][3].z)
                                    : make_float4(blk[i][0].w, blk[i][1].w, blk[i][2].w, blk[i][3].w);
            const float4 hv = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
            const uint32_t off = (kg >> 3) * kSlabK + d * 128 + (((kg & 7) ^ (d & 7)) << 4);
            *reinterpret_cast<float4*>(vh + off) = hv;
            *reinterpret_cast<float4*>(vl + off) = make_float4(v.x - hv.x, v.y - hv.y, v.z - hv.z, v.w - hv.w);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->v_ready[vs]);
      }
      if (!ok) break;
    }
  } else if (warp == 14) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuer: S
      // S(h) = Q K^T, the two small products first, then the high one.  Its
      // buffer last held S(h-3) and then P(h-3)'s high parts, read by PV(h-3)
      // from the other issuer: that PV has completed before S(h) is issued.
      const uint64_t kd0 = sdesc_sw128(smem_u32(smem) + kOffK, 16, 1024);  // descriptor of key stage 0
      uint32_t n = 0, h = 0;  // units, halves
      bool ok = true;
      for (;; ++n) {
        const int slot = n & 1;
        if (!(ok = wait(&sh->unit_full[slot], (n >> 1) & 1))) break;
        const UnitInfo inf = sh->info[slot];
        mbar_arrive(&sh->unit_empty[slot]);
        if (inf.u < 0) break;
        for (int k = 0; k < inf.nsub; ++k, ++h) {
          const uint32_t st = h % kKStages;
          if (!(ok = wait(&sh->k_ready[st], (h / kKStages) & 1))) break;
          if (k == 0 && !(ok = wait(&sh->q_ready, n & 1))) break;
          if (h >= kSBufs && !(ok = wait(&sh->pv_buf[h % kSBufs], ((h - kSBufs) / kSBufs) & 1))) break;
          tc_fence_after();
          // descriptors advance by (byte offset >> 4) in their address field
          const uint64_t kd = kd0 + ((st * 2 * kHalfBytes) >> 4);
          const uint32_t tS = tmem + kColS + 64 * (h % kSBufs);
#pragma unroll 1
          for (int q = 0; q < 3; ++q) {
            const uint32_t a = q == 0 ? tmem + kColQl : tmem + kColQh;
            const uint64_t b = kd + ((q == 1 ? kHalfBytes : 0u) >> 4);
#pragma unroll
            for (int ks = 0; ks < kHead / 8; ++ks)
              mma_tf32_ts(tS, a + ks * 8, b + (((ks >> 2) * kSlabK + (ks & 3) * 32) >> 4), (q | ks) != 0 ? 1u : 0u);
          }
          tc_commit(&sh->s_full[h % kSBufs]);
          tc_commit(&sh->k_empty[st]);
          if (k + 1 == inf.nsub) tc_commit(&sh->q_free);
        }
        if (!ok) break;
      }
      if (*abort_flag) {  // every MMA this thread issued completes before TMEM is freed
        tc_commit(&sh->drain[0]);
        mbar_wait(&sh->drain[0], 0);
      }
    }
    __syncwarp();
  } else if (warp == 15) {
    if (lane == 0) {
      // ----------------------------------------------------- MMA issuer: PV
      // O += P(h) V(h), the two small products first, then the high one; a
      // unit's first half overwrites O once the epilogue of the unit before
      // it has read O
      const uint64_t vd0 = sdesc_sw128(smem_u32(smem) + kOffV, 16, 1024);  // descriptor of V^T stage 0
      uint32_t n = 0, h = 0;
      bool ok = true;
      for (;; ++n) {
        const int slot = n & 1;
        if (!(ok = wait(&sh->unit_full[slot], (n >> 1) & 1))) break;
        const UnitInfo inf = sh->info[slot];
        mbar_arrive(&sh->unit_empty[slot]);
        if (inf.u < 0) break;
        for (int k = 0; k < inf.nsub; ++k, ++h) {
          const uint32_t st = h % kVStages;
          if (!(ok = wait(&sh->p_full[h % kSBufs], (h / kSBufs) & 1))) break;
          if (!(ok = wait(&sh->v_ready[st], (h / kVStages) & 1))) break;
          if (k == 0 && n > 0 && !(ok = wait(&sh->o_free, (n - 1) & 1))) break;
          tc_fence_after();
          const uint64_t vd = vd0 + ((st * 2 * kHalfBytes) >> 4);
          const uint32_t ph = tmem + kColS + 64 * (h % kSBufs), pl = tmem + kColPl + 64 * (h & 1);
#pragma unroll 1
          for (int q = 0; q < 3; ++q) {
            const uint32_t a = q == 0 ? pl : ph;
            const uint64_t b = vd + ((q == 1 ? kHalfBytes : 0u) >> 4);
#pragma unroll
            for (int ks = 0; ks < kSub / 8; ++ks)
              mma_tf32_ts(tmem + kColO, a + ks * 8, b + (((ks >> 2) * kSlabK + (ks & 3) * 32) >> 4),
                          (k > 0 || (q | ks) != 0) ? 1u : 0u);
          }
          tc_commit(&sh->pv_buf[h % kSBufs]);
          tc_commit(&sh->v_empty[st]);
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        tc_commit(&sh->drain[1]);
        mbar_wait(&sh->drain[1], 0);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int c = warp >> 2;                    // key columns 32c .. 32c + 31 of each half; O columns likewise
    const int r = (warp & 3) * 32 + lane;       // row in the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t h = 0, xc = 0;
    bool ok = true;
    UnitInfo inf;
    // The unit's queries, rotated and scaled, split into TMEM: this thread
    // takes rotation pairs (t, t + 32) for t in 16c .. 16c + 15 of row r.
    // Every softmax warp passes the same named barriers in the same order: per
    // unit two over all eight warps (in load_unit), per half and at the
    // epilogue one over the two warps of the same rows.  A failed wait is
    // carried to the next eight-warp barrier, where all leave together.
    auto load_unit = [&](uint32_t m, bool good) -> bool {
      const int slot = m & 1;
      good = __all_sync(0xffffffffu, good && wait(&sh->unit_full[slot], (m >> 1) & 1));
      if (named_bar_or(1, 256, !good)) {
        inf.u = -1;
        return false;
      }
      inf = sh->info[slot];
      named_bar_or(1, 256, false);  // every thread has its copy of the unit
      if (tid == 0) mbar_arrive(&sh->unit_empty[slot]);
      if (inf.u < 0) return true;
      const int pos = inf.q0 + r;
      const bool rot = pos < inf.L;  // (a row past the sequence's end is never written out)
      const float* crow = p.cos_t + static_cast<size_t>(rot ? pos : 0) * kHalf + 16 * c;
      const float* srow = p.sin_t + static_cast<size_t>(rot ? pos : 0) * kHalf + 16 * c;
      float4 cs[4], sn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        cs[e] = __ldg(reinterpret_cast<const float4*>(crow) + e);
        sn[e] = __ldg(reinterpret_cast<const float4*>(srow) + e);
      }
      good = __all_sync(0xffffffffu, wait(&sh->q_raw_full, m & 1));
      // the previous unit's S MMAs have read its Q columns
      if (m > 0) good = __all_sync(0xffffffffu, good && wait(&sh->q_free, (m - 1) & 1));
      if (!good) return false;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // pairs 16c + 8 half .. + 7
        uint32_t hlo[8], hhi[8], llo[8], lhi[8];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int e = 2 * half + e2;
          // 16-byte chunk 4c + e of the row in each slab (128-byte swizzle)
          const uint32_t off = r * 128 + (((4 * c + e) ^ (r & 7)) << 4);
          const float4 a4 = *reinterpret_cast<const float4*>(smem + kOffQ + off);
          const float4 b4 = *reinterpret_cast<const float4*>(smem + kOffQ + kSlabQ + off);
          const float xa[4] = {a4.x, a4.y, a4.z, a4.w}, xb[4] = {b4.x, b4.y, b4.z, b4.w};
          const float cc[4] = {cs[e].x, cs[e].y, cs[e].z, cs[e].w}, ss[4] = {sn[e].x, sn[e].y, sn[e].z, sn[e].w};
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            float ya = xa[f], yb = xb[f];
            if (rot) rope_pair(xa[f], xb[f], cc[f], ss[f], ya, yb);
            ya *= p.qmul;
            yb *= p.qmul;
            const float ha = tf32_hi(ya), hb = tf32_hi(yb);
            hlo[4 * e2 + f] = __float_as_uint(ha);
            llo[4 * e2 + f] = __float_as_uint(ya - ha);
            hhi[4 * e2 + f] = __float_as_uint(hb);
            lhi[4 * e2 + f] = __float_as_uint(yb - hb);
          }
        }
        const uint32_t col = 16 * c + 8 * half;
        tmem_st8(tmem + kColQh + col + lane_off, hlo);
        tmem_st8(tmem + kColQh + 32 + col + lane_off, hhi);
        tmem_st8(tmem + kColQl + col + lane_off, llo);
        tmem_st8(tmem + kColQl + 32 + col + lane_off, lhi);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh->q_raw_empty);  // the raw tile may take the next unit's queries
        mbar_arrive(&sh->q_ready);
      }
      return true;
    };
    // One pass per unit: its queries into TMEM (unit m), the previous unit's
    // epilogue, then this unit's halves.  The queries of unit m go into TMEM
    // once every S of unit m-1 is done, so its first S overlaps unit m-1's
    // last PV.
    UnitInfo cur;
    cur.u = -1;
    int i = 0;
    bool row_ok = false;
    float l = 0.f;
    for (uint32_t m = 0;; ++m) {
      ok = load_unit(m, ok);
      if (cur.u >= 0) {
        // epilogue: the row sums of both warps, then the unit's last PV, then O
        // / l in this warp's 32 output columns
        sh->xl[c][r] = l;
        if (named_bar_or(2 + (warp & 3), 64, !ok)) ok = false;  // (the next load_unit barrier ends the loop)
        const float inv = 1.f / (l + sh->xl[1 - c][r]);
        // (the partner reads xl[c] before its next barrier with this thread,
        // which comes before xl is written again)
        ok = __all_sync(0xffffffffu, ok && wait(&sh->pv_buf[(h - 1) % kSBufs], ((h - 1) / kSBufs) & 1));
        tc_fence_after();
        if (ok) {
          uint32_t ov[32];
          tmem_ld32_wait(tmem + kColO + 32 * c + lane_off, ov);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->o_free);
          if (row_ok) {
            float* dst = p.out + static_cast<size_t>(cur.row0 + i) * p.heads * kHead + cur.h * kHead + 32 * c;
#pragma unroll
            for (int d = 0; d < 32; d += 4)
              *reinterpret_cast<float4*>(dst + d) =
                  make_float4(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv,
                              __uint_as_float(ov[d + 2]) * inv, __uint_as_float(ov[d + 3]) * inv);
          }
        }
      }
      if (inf.u < 0) break;
      cur = inf;
      i = cur.q0 + r;
      row_ok = i < cur.L;
      // Online softmax with a lazily moved reference max m_ref: P = 2^(S -
      // m_ref); O and the row sum l stay relative to m_ref, which moves --
      // rescaling both -- only when a row's max exceeds it by more than 2^8.
      // Both warps of a row hold the same m_ref; each sums its own columns.
      float m_ref = kNone;
      l = 0.f;
      for (int k = 0; k < cur.nsub; ++k, ++h) {
        ok = __all_sync(0xffffffffu, ok && wait(&sh->s_full[h % kSBufs], (h / kSBufs) & 1));
        tc_fence_after();
        const uint32_t tS = tmem + kColS + 64 * (h % kSBufs) + 32 * c + lane_off;
        const uint32_t tPl = tmem + kColPl + 64 * (h & 1) + 32 * c + lane_off;
        uint32_t sv[32];
        if (ok) tmem_ld32_wait(tS, sv);
        const int hf = cur.hb + k, k0 = hf * kSub + 32 * c;  // this warp's first key
        const bool full = !kNarrow && hf >= cur.ffb && hf < cur.ffe;
        // visible keys of this row among this warp's 32: columns [lo, hi],
        // one bit each in vis
        uint32_t vis = ~0u;
        if (!full) {
          int lo = 0, hi = min(31, cur.L - 1 - k0);
          if (p.causal) hi = min(hi, i - k0);
          if (p.window >= 0) {
            lo = max(0, i - p.window - k0);
            hi = min(hi, i + p.window - k0);
          }
          if (!row_ok) hi = -1;
          const uint32_t upto_hi = hi < 0 ? 0u : (2u << min(hi, 31)) - 1u;
          const uint32_t below_lo = lo <= 0 ? 0u : (lo >= 32 ? ~0u : (1u << lo) - 1u);
          vis = upto_hi & ~below_lo;
        }
        // the maximum over the visible columns (kNone when there are none);
        // masked columns are left out, and get probability 0 below
        float m8[8];
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q) m8[q] = fmaxf(__uint_as_float(sv[4 * q]), __uint_as_float(sv[4 * q + 1]));
#pragma unroll
          for (int q = 0; q < 8; ++q)
            m8[q] = fmax3(m8[q], __uint_as_float(sv[4 * q + 2]), __uint_as_float(sv[4 * q + 3]));
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) m8[q] = kNone;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if ((vis >> j) & 1u) m8[j >> 2] = fmaxf(m8[j >> 2], __uint_as_float(sv[j]));
        }
        float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        // the row's maximum over both warps' columns
        float* xb = &sh->xch[xc & 1][0][0];
        ++xc;
        xb[c * kBM + r] = mx;
        // the two warps of these rows only (barrier 2 + lane quarter, 64 threads)
        if (named_bar_or(2 + (warp & 3), 64, !ok)) {
          ok = false;  // (all eight warps learn of it at load_unit's barrier)
          break;
        }
        mx = fmaxf(mx, xb[(1 - c) * kBM + r]);
        float alpha = 1.f;
        if (mx > m_ref + kLazy) {
          if (m_ref != kNone) alpha = fast_exp2(m_ref - mx);
          m_ref = mx;
        }
        // P = 2^(S - m_ref) for the visible columns, 0 for the masked ones
        // (while the row has no visible key yet, m_ref = kNone, its reference
        // is taken as 0)
        const float mr = m_ref == kNone ? 0.f : m_ref;
        // P-low buffer h mod 2 was last read by PV(h-2)
        if (h >= 2) {
          ok = __all_sync(0xffffffffu, wait(&sh->pv_buf[(h - 2) % kSBufs], ((h - 2) / kSBufs) & 1));
          tc_fence_after();
        }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 16 columns at a time: P high over S, P low beside
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float pe = (vis >> (16 * q + e)) & 1u ? fast_exp2(__uint_as_float(sv[16 * q + e]) - mr) : 0.f;
            const float hv = tf32_hi(pe);
            s4[e & 3] += pe;
            ph[e] = __float_as_uint(hv);
            pl[e] = __float_as_uint(pe - hv);
          }
          tmem_st16(tS + 16 * q, ph);
          tmem_st16(tPl + 16 * q, pl);
        }
        l = l * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
        // O is rescaled once PV(h-1) has accumulated into it (and before
        // PV(h), which waits for this half's P)
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          ok = __all_sync(0xffffffffu, ok && wait(&sh->pv_buf[(h - 1) % kSBufs], ((h - 1) / kSBufs) & 1));
          tc_fence_after();
          if (ok) {
            uint32_t ov[32];
            tmem_ld32_wait(tmem + kColO + 32 * c + lane_off, ov);
#pragma unroll
            for (int d = 0; d < 32; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
            tmem_st32(tmem + kColO + 32 * c + lane_off, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&sh->p_full[h % kSBufs]);
      }
    }
  }

  // Wind down: after an abort the producer and the issuer have waited
  // (bounded) for their own copies and MMAs in flight; then TMEM is freed.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kT3Cols);
  }
}

}  // namespace

cudaError_t launch_prefill_3xtf32(const CUtensorMap* qkv_map, int heads, int kv_heads, int window, int causal,
                                  float scale, const float* cos_t, const float* sin_t, float* out, void* ws,
                                  int32_t* dev_status, cudaStream_t st) {
  static int configured[2][64] = {};
  const bool narrow = window >= 0 && window <= 64;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (dev >= 64 || !configured[narrow][dev]) {
    const void* fn = narrow ? reinterpret_cast<const void*>(prefill_3xtf32_kernel<true>)
                            : reinterpret_cast<const void*>(prefill_3xtf32_kernel<false>);
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kT3Smem)) != cudaSuccess)
      return e;
    if (dev < 64) configured[narrow][dev] = 1;
  }
  T3Params prm;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.window = window;
  prm.causal = causal;
  prm.qmul = scale * 1.4426950408889634f;
  prm.cos_t = cos_t;
  prm.sin_t = sin_t;
  prm.out = out;
  prm.hdr = static_cast<WsHeader*>(ws);
  prm.pairs = ws_pairs(ws);
  prm.dev_status = dev_status;
  // launched with programmatic stream serialization: its prologue overlaps
  // the kernels before it, whose results the producer waits for (griddep_wait)
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
  return narrow ? cudaLaunchKernelEx(&cfg, prefill_3xtf32_kernel<true>, *qkv_map, prm)
                : cudaLaunchKernelEx(&cfg, prefill_3xtf32_kernel<false>, *qkv_map, prm);
}

}  // namespace kime
