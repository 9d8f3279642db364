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
// Split-KV, streamed: the keys 0..=pos[s] of a (sequence, kv head) are cut
// into chunks of 128 and the chunks into work items of up to 16 (2048 keys).
// Persistent CTAs (three per SM) take items from shared counters.  In each
// CTA one producer warp claims items, rotates their q heads into an item slot
// and streams their chunks' K and V tiles (TMA, 128-byte swizzle) through a
// 2-stage ring to four consumer warps, which reduce each chunk on the tensor
// cores: S = q K^T for all G q heads of the kv group (the GQA fold: the cache
// is read once per kv head), online softmax per head, O += P V.  Memory never
// waits for a CTA to set up, compute or merge: the SM's other CTAs keep their
// copies in flight.  Each item ends in a part (m, l, o[64]) per q head
// (base-2 logits); the last part of a (sequence, kv head) to finish -- found
// with an atomic ticket, no waiting -- merges the parts:
// m = max m_c, l = sum l_c 2^(m_c-m), o = sum o_c 2^(m_c-m) / l.
#include <algorithm>

#include "kime_common.cuh"

#ifdef KIME_PHASE_PROFILE
__device__ unsigned long long g_kime_dec_phase[16];  // producer 0.., consumer group 0 8..
__device__ unsigned long long g_kime_dec_span[2 * 1024];  // per CTA: start, end (globaltimer)
#endif

namespace kime {

namespace {

constexpr int kAppendThreads = 128;
constexpr uint32_t kStageBytes = 2 * kDecChunk * kHead * 2;  // K and V of one chunk
constexpr int kPartialFloats = 68;              // m, l, o[64], 2 pad
constexpr int kItemChunks = kDecItemChunks;      // chunks per work item
constexpr int kMergeBlock = 64;                 // parts weighted at once by the final merge
// Three CTAs per SM, each a producer warp and one consumer group of 4 warps
// with a 2-stage chunk ring: while one CTA merges an item, the other two keep
// the SM's copies in flight.  In the group, warp w takes keys 32 w .. 32 w + 31
// of the chunk on the tensor cores (mma.sync m16n8k16, bf16 in, f32
// accumulate): S = q K^T with the kv group's q heads as rows (padded to 16),
// then P V with P from registers.
template <int G>
struct DecCfg {
  static constexpr int n_grp = 1;                              // consumer groups (dec_groups_for)
  static constexpr int warps = 4 * n_grp;                      // consumer warps
  static constexpr int consumers = warps * 32;
  static constexpr int threads = consumers + 32;               // plus the producer warp
  static constexpr int ring = 2;                               // stages in all
  static constexpr int ctas_per_sm = 3;
  static constexpr int sub_ring = ring / n_grp;                // stages per group
};
constexpr int kGroupThreads = 128;

struct DecItem {
  int32_t s, g, c0, c1, P, n_c;  // s < 0: no more items
};

// Shared memory of one decode CTA (offsets in bytes).
template <int G>
struct DecLayout {
  using Cfg = DecCfg<G>;
  static constexpr int kRing = Cfg::ring;
  static constexpr uint32_t ring = 0;
  static constexpr uint32_t q = ring + kRing * kStageBytes;             // [2][G][64] f32
  static constexpr uint32_t info = q + 2 * G * kHead * 4;               // [2] DecItem
  // per consumer group: the part combine ([4][G][64] o, [4][G] m, [4][G] l)
  // and, after it, the final merge ([G][128] maxima, [2G] M and L,
  // [kMergeBlock][G] weights) share one region
  static constexpr uint32_t red = info + 64;
  static constexpr uint32_t red_bytes = 4 * G * (kHead + 2) * 4;
  static constexpr uint32_t merge_bytes = G * (kGroupThreads + 2 + kMergeBlock) * 4;
  static constexpr uint32_t red_stride = ((red_bytes > merge_bytes ? red_bytes : merge_bytes) + 15) / 16 * 16;
  static constexpr uint32_t bars = red + Cfg::n_grp * red_stride;  // full, empty, item_full, item_empty
  static constexpr uint32_t flags = bars + (2 * kRing + 4) * 8;         // abort, last
  static constexpr uint32_t bytes = flags + 16 + 1024;  // abort, one "last part" flag per group; alignment slack
};

// Warp-level tensor-core MMA m16n8k16, bf16 inputs, f32 accumulate (D += A B).
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// Byte offset of 16-byte piece j of row r in a tile written by TMA with the
// 128-byte swizzle (rows of 128 bytes, tile 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// Barrier 1 among the consumer warps only (N threads), with an OR vote.
template <int N>
__device__ __forceinline__ bool bar_or_consumers(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(N)
      : "memory");
  return r != 0;
}
template <int N>
__device__ __forceinline__ void bar_consumers() {
  asm volatile("barrier.cta.sync 1, %0;" ::"n"(N) : "memory");
}
// Barrier 2 + grp among the 128 threads of one consumer group, with an OR vote.
__device__ __forceinline__ bool bar_or_group(int grp, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(2 + grp), "n"(kGroupThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_group(int grp) {
  asm volatile("barrier.cta.sync %0, %1;" ::"r"(2 + grp), "n"(kGroupThreads) : "memory");
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

struct DecPlan {
  int32_t next, n_items, pad[2];  // work counter, items in the list
};

// The work list of one decode launch (one CTA): item k of (s, g) covers chunks
// I k .. min(I k + I, n_c) - 1 (I = kItemChunks) of keys 0..=pos[s].  Full
// items come first, then
// the shorter last items by decreasing size (a counting sort on the chunk
// count), so the CTAs that take the last items finish soon after the others.
// Item 0 of (s, g) number b < n_static is not listed: CTA b of the decode
// kernel takes it at once, before this list is ready.  Also zeroes the
// tickets and reports positions outside [0, min(cap, rope_len)) (those
// sequences get no items).
__global__ void __launch_bounds__(1024)
    decode_plan_kernel(const int32_t* __restrict__ pos, int n_seqs, int kv_heads, int cap, int rope_len,
                       int n_static, DecPlan* plan, int32_t* __restrict__ tickets, int4* __restrict__ items,
                       int32_t* dev_status) {
  __shared__ int hist[kItemChunks + 1], cursor[kItemChunks + 1];
  __shared__ int s_bad;
  griddep_launch_dependents();  // the decode kernel sets itself up meanwhile
  if (threadIdx.x <= kItemChunks) hist[threadIdx.x] = 0;
  if (threadIdx.x == 0) s_bad = 0;
  for (int i = threadIdx.x; i < n_seqs * kv_heads; i += blockDim.x) tickets[i] = 0;
  __syncthreads();
  auto chunks_of = [&](int s) -> int {
    const int P = pos[s];
    if (P < 0 || P >= cap || P >= rope_len) return -1;
    return (P + kDecChunk) / kDecChunk;
  };
  for (int s = threadIdx.x; s < n_seqs; s += blockDim.x) {
    const int n_c = chunks_of(s);
    if (n_c < 0) {
      s_bad = 1;
      continue;
    }
    for (int g = 0; g < kv_heads; ++g)  // item 0 of the first n_static (s, g) is not listed
      for (int k = s * kv_heads + g < n_static ? 1 : 0; k * kItemChunks < n_c; ++k)
        atomicAdd(&hist[min(kItemChunks, n_c - k * kItemChunks)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int sz = kItemChunks; sz >= 1; --sz) {
      cursor[sz] = acc;
      acc += hist[sz];
    }
    plan->next = 0;
    plan->n_items = acc;
    if (s_bad) report(dev_status, ST_BAD_POS);
  }
  __syncthreads();
  for (int s = threadIdx.x; s < n_seqs; s += blockDim.x) {
    const int n_c = chunks_of(s);
    if (n_c < 0) continue;
    const int P = pos[s];
    for (int g = 0; g < kv_heads; ++g)
      for (int k = s * kv_heads + g < n_static ? 1 : 0; k * kItemChunks < n_c; ++k)
        items[atomicAdd(&cursor[min(kItemChunks, n_c - k * kItemChunks)], 1)] = make_int4(s, g, k, P);
  }
}

// kAppend: the consumer warps of the item holding row pos[s] (its last chunk)
// also perform the KV append of kv_append_kernel for their kv head (the same
// float32 rotation and rounding): they write the row to the caches and over
// the stale copy in the stage, so append and attention take one launch.  No
// other CTA reads that row.
template <int G, bool kAppend>
__global__ void __launch_bounds__(DecCfg<G>::threads, DecCfg<G>::ctas_per_sm)
    decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                  const uint16_t* __restrict__ qkv_new, const int32_t* __restrict__ pos, int n_seqs, int heads,
                  int kv_heads, int cap, float scale_log2, const float* __restrict__ cos_t,
                  const float* __restrict__ sin_t, int rope_len, uint16_t* __restrict__ k_cache,
                  uint16_t* __restrict__ v_cache, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ partials, int32_t* __restrict__ tickets, DecPlan* plan,
                  const int4* __restrict__ items, int max_items, int n_static, int32_t* dev_status) {
  using Lay = DecLayout<G>;
  using Cfg = DecCfg<G>;
  constexpr int kRing = Cfg::ring, kDecWarps = Cfg::warps;
  constexpr int kGrp = Cfg::n_grp, kSub = Cfg::sub_ring;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled TMA tiles need a 1024-byte aligned base
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* qslot = reinterpret_cast<float*>(smem + Lay::q);
  DecItem* info = reinterpret_cast<DecItem*>(smem + Lay::info);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::bars);
  uint64_t* empty = full + kRing;
  uint64_t* item_full = empty + kRing;
  uint64_t* item_empty = item_full + 2;
  volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + Lay::flags);
  int32_t* s_last = reinterpret_cast<int32_t*>(smem + Lay::flags) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);

#ifdef KIME_PHASE_PROFILE
  if (tid == 0 && blockIdx.x < 1024) g_kime_dec_span[2 * blockIdx.x] = globaltimer();
#endif
  if (tid == 0) {
    tma_prefetch_map(&k_map);
    tma_prefetch_map(&v_map);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);  // the four warps of the stage's group
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(dev_status, ST_TIMEOUT);
    return false;
  };

  if (warp == kDecWarps) {
    // ------------------------------------------------------------ producer warp
    uint32_t it = 0, cs = 0;  // items published, chunks issued
    bool ok = true;
    PHASE_DECL(5);
    // The first item of CTA b < n_static is item 0 of (s, g) number b, taken
    // at once; the rest come one at a time from the plan kernel's list.
    bool first = blockIdx.x < n_static, listed = false;
    int n_items = 0;
    for (;;) {
      int4 rec;
      if (first) {
        first = false;
        const int sg = blockIdx.x, s0 = sg / kv_heads, P0 = __ldg(pos + s0);
        if (P0 < 0 || P0 >= cap || P0 >= rope_len) continue;  // reported by the plan kernel
        rec = make_int4(s0, sg - s0 * kv_heads, 0, P0);
      } else {
        if (!listed) {
          griddep_wait();  // the work list of the plan kernel before this one
          n_items = plan->n_items;
          listed = true;
        }
        int idx = 0;
        if (lane == 0) idx = atomicAdd(&plan->next, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx >= n_items) break;
        rec = items[idx];
      }
      PHASE(0);
      {
        const int is = rec.x, ig = rec.y, ik = rec.z, iP = rec.w;
        const int inc = (iP + kDecChunk) / kDecChunk;  // chunks of keys 0..=P
        const int slot = it & 1;
        PHASE(2);
        if (lane == 0) ok = wait(&item_empty[slot], ((it >> 1) & 1) ^ 1);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
        PHASE(1);
        // the item's q heads, rotated at P (lane t owns the pair t, t+32), times
        // scale * log2(e)
        {
          const float c = __ldg(cos_t + static_cast<size_t>(iP) * kHalf + lane);
          const float sn = __ldg(sin_t + static_cast<size_t>(iP) * kHalf + lane);
          float* qd = qslot + slot * G * kHead;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const uint16_t* xq = qkv_new + static_cast<size_t>(is) * W + (ig * G + hh) * kHead;
            const float a = __uint_as_float(static_cast<uint32_t>(__ldg(xq + lane)) << 16);
            const float b = __uint_as_float(static_cast<uint32_t>(__ldg(xq + lane + kHalf)) << 16);
            float ya, yb;
            rope_pair(a, b, c, sn, ya, yb);
            qd[hh * kHead + lane] = ya * scale_log2;
            qd[hh * kHead + lane + kHalf] = yb * scale_log2;
          }
        }
        const int c0 = ik * kItemChunks, c1 = min(c0 + kItemChunks, inc);
        if (lane == 0) info[slot] = DecItem{is, ig, c0, c1, iP, inc};
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_full[slot]);
        ++it;
        PHASE(2);
        if (lane == 0) {
          for (int c = c0; c < c1; ++c, ++cs) {
            // chunk cs -> group cs % kGrp, that group's fill number rp
            const uint32_t rp = cs / kGrp;
            const int st = (cs % kGrp) * kSub + rp % kSub;
            PHASE(4);
            if (!(ok = wait(&empty[st], ((rp / kSub) & 1) ^ 1))) break;
            PHASE(3);
            // whole 128-row tiles, 128-byte swizzle: rows past pos[s] are
            // masked (K) and zeroed (V) by the consumers
            const int y = (is * kv_heads + ig) * cap + c * kDecChunk;
            mbar_arrive_expect_tx(&full[st], kStageBytes);
            tma_load_2d(smem + Lay::ring + st * kStageBytes, &k_map, &full[st], 0, y);
            tma_load_2d(smem + Lay::ring + st * kStageBytes + kStageBytes / 2, &v_map, &full[st], 0, y);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
      }
    }
    if (ok) {  // no more items
      const int slot = it & 1;
      if (lane == 0 && wait(&item_empty[slot], ((it >> 1) & 1) ^ 1)) {
        info[slot].s = -1;
        mbar_arrive(&item_full[slot]);
      }
    }
    cs = __shfl_sync(0xffffffffu, cs, 0);
    if (*abort_flag && lane == 0)  // the copies this warp issued land before the CTA leaves
      for (uint32_t x = (cs > kRing ? cs - kRing : 0); x < cs; ++x) {  // the last fill of every stage
        const uint32_t rp = x / kGrp;
        mbar_wait(&full[(x % kGrp) * kSub + rp % kSub], (rp / kSub) & 1);
      }
    PHASE(4);
    PHASE_FLUSH(g_kime_dec_phase, 0, lane == 0);
  } else {
    // ------------------------------------------------------------ consumer groups
    // Each group of 4 warps runs on its own: its chunks of every item, then its
    // own part (m, l, o) of the item, so one group's merge overlaps the other
    // groups' chunks.  Parts of (s, g): items x groups; the last to finish
    // (atomic ticket) merges them.
    const int cg = warp >> 2, gtid = tid & (kGroupThreads - 1);  // consumer group, thread in it
    const int gw = warp & 3;                                     // warp in the group
    float* red_o = reinterpret_cast<float*>(smem + Lay::red + cg * Lay::red_stride);  // [4][G][64]
    float* red_m = red_o + 4 * G * kHead;                                           // [4][G]
    float* red_l = red_m + 4 * G;                                                   // [4][G]
    int32_t* g_last = s_last + cg;
    uint32_t it = 0, cs = 0;
    PHASE_DECL(6);
    for (;; ++it) {
      const int slot = it & 1;
      PHASE(4);
      bool ok = wait(&item_full[slot], (it >> 1) & 1);
      if (bar_or_group(cg, !ok)) break;
      const DecItem item = info[slot];
      if (item.s < 0) break;
      // q as the A operand: rows = the G q heads (rows >= G and 8..15 are zero),
      // 4 k-steps of 16 dims; thread (gq = lane / 4, tq = lane % 4) holds row gq,
      // dims 16 ks + 2 tq (+1) and 16 ks + 8 + 2 tq (+1)
      const int gq = lane >> 2, tq = lane & 3;
      uint32_t qa[4][4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const float* qr = qslot + (slot * G + (gq < G ? gq : 0)) * kHead + ks * 16 + 2 * tq;
        qa[ks][0] = gq < G ? pack_bf16x2(qr[0], qr[1]) : 0u;
        qa[ks][2] = gq < G ? pack_bf16x2(qr[8], qr[9]) : 0u;
        qa[ks][1] = qa[ks][3] = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);  // this warp has its q
      PHASE(0);
      const int s = item.s, g = item.g, P = item.P;
      // this warp: keys 32 gw .. 32 gw + 31 of every chunk of the group; its
      // running (m, l) for row gq and O (rows gq, gq + 8) as 8 n-tiles of dims
      float m_run = kNone, l_run = 0.f;  // kNone: no key yet (finite, below every logit)
      float oacc[8][4];
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) oacc[nd][0] = oacc[nd][1] = oacc[nd][2] = oacc[nd][3] = 0.f;
      const int kbase = gw * 32;
      for (int c = item.c0; c < item.c1; ++c, ++cs) {
        if (static_cast<int>(cs % kGrp) != cg) continue;  // another group's chunk
        const uint32_t rp = cs / kGrp;
        const int st = cg * kSub + rp % kSub, nk = min(kDecChunk, P + 1 - c * kDecChunk);
        uint8_t* stage = smem + Lay::ring + st * kStageBytes;
        PHASE(5);
        ok = wait(&full[st], (rp / kSub) & 1);
        if (bar_or_group(cg, !ok)) { ok = false; break; }  // the whole group leaves the item
        PHASE(2);
        const bool patch = kAppend && c == item.n_c - 1;
        if (nk < kDecChunk || patch) {
          uint16_t* Vz = reinterpret_cast<uint16_t*>(stage + kStageBytes / 2);
          // rows past pos[s] come from other cache rows: zero V there (a NaN
          // would reach O through a zero probability); K is masked below
          for (int e = nk * 8 + gtid; e < kDecChunk * 8; e += kGroupThreads)
            reinterpret_cast<uint4*>(Vz)[e] = make_uint4(0u, 0u, 0u, 0u);
          if (patch) {
            // this chunk holds row P: write the appended k (rotated at P) and v
            // of kv head g to the caches and over the stale copy in the stage
            const int prow = P - c * kDecChunk;  // row P within the chunk
            uint16_t* ks = reinterpret_cast<uint16_t*>(stage);
            const uint16_t* row = qkv_new + static_cast<size_t>(s) * W;
            const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
            if (gtid < kHalf) {
              const uint16_t* xk = row + (heads + g) * kHead;
              const float a = __uint_as_float(static_cast<uint32_t>(xk[gtid]) << 16);
              const float b = __uint_as_float(static_cast<uint32_t>(xk[gtid + kHalf]) << 16);
              float ya, yb;
              rope_pair(a, b, cos_t[static_cast<size_t>(P) * kHalf + gtid],
                        sin_t[static_cast<size_t>(P) * kHalf + gtid], ya, yb);
              const uint32_t w2 = pack_bf16x2(ya, yb);
              const uint16_t lo = static_cast<uint16_t>(w2 & 0xffffu), hi = static_cast<uint16_t>(w2 >> 16);
              k_cache[dst + gtid] = lo;
              k_cache[dst + gtid + kHalf] = hi;
              ks[(sw128(prow, gtid >> 3) >> 1) + (gtid & 7)] = lo;
              ks[(sw128(prow, (gtid + kHalf) >> 3) >> 1) + (gtid & 7)] = hi;
            } else if (gtid < kHalf + kHead) {
              const int t = gtid - kHalf;
              const uint16_t v = row[(heads + kv_heads + g) * kHead + t];
              v_cache[dst + t] = v;
              Vz[(sw128(prow, t >> 3) >> 1) + (t & 7)] = v;
            }
          }
          fence_proxy_async_smem();  // the stage is refilled by TMA later
          bar_group(cg);
        }
        const uint32_t sK = smem_u32(stage), sV = sK + kStageBytes / 2;
        // S = q K^T for this warp's 32 keys: 4 n-tiles of 8 keys x 4 k-steps
        float sacc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
          const int key = kbase + nt * 8 + (lane & 7);  // the row this lane addresses
          uint32_t b0[4], b1[4];
          ldsm_x4(b0, sK + sw128(key, lane >> 3));        // dims pieces 0..3
          ldsm_x4(b1, sK + sw128(key, 4 + (lane >> 3)));  // dims pieces 4..7
          mma_bf16(sacc[nt], qa[0], b0[0], b0[1]);
          mma_bf16(sacc[nt], qa[1], b0[2], b0[3]);
          mma_bf16(sacc[nt], qa[2], b1[0], b1[1]);
          mma_bf16(sacc[nt], qa[3], b1[2], b1[3]);
        }
        // row gq: keys kbase + 8 nt + 2 tq (+1); keys past pos[s] are left
        // out of the maximum and get probability 0 below (no -inf is formed)
        float mloc = kNone;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int k0 = kbase + nt * 8 + 2 * tq;
          if (k0 < nk) mloc = fmaxf(mloc, sacc[nt][0]);
          if (k0 + 1 < nk) mloc = fmaxf(mloc, sacc[nt][1]);
        }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        if (mloc > m_run) {  // the running max grows: rescale l and O
          const float alpha = fast_exp2(m_run - mloc);  // 0 while m_run is still kNone
          l_run *= alpha;
#pragma unroll
          for (int nd = 0; nd < 8; ++nd) {
            oacc[nd][0] *= alpha;
            oacc[nd][1] *= alpha;
          }
          m_run = mloc;
        }
        const float m_use = m_run == kNone ? 0.f : m_run;
        // P = 2^(S - m) rounded to bf16 (the row sum takes the rounded values,
        // so the weights and their normalisation agree), as the A operand of
        // P V: k-step kk = n-tiles 2kk (pieces 0) and 2kk + 1 (pieces 2)
        uint32_t pa[2][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int k0 = kbase + nt * 8 + 2 * tq;
          const uint32_t pw = pack_bf16x2(k0 < nk ? fast_exp2(sacc[nt][0] - m_use) : 0.f,
                                          k0 + 1 < nk ? fast_exp2(sacc[nt][1] - m_use) : 0.f);
          l_run += bf16lo(pw) + bf16hi(pw);
          pa[nt >> 1][(nt & 1) * 2] = pw;
          pa[nt >> 1][(nt & 1) * 2 + 1] = 0u;
        }
        // O += P V: 2 k-steps of 16 keys x 8 n-tiles of 8 dims; V through
        // transposing loads (rows = keys)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int key = kbase + kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
          for (int nd = 0; nd < 8; nd += 2) {
            uint32_t bv[4];
            ldsm_x4_t(bv, sV + sw128(key, nd + (lane >> 4)));
            mma_bf16(oacc[nd], pa[kk], bv[0], bv[1]);
            mma_bf16(oacc[nd + 1], pa[kk], bv[2], bv[3]);
          }
        }
        if (patch || nk < kDecChunk) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
        PHASE(3);
      }
      if (!ok) break;
      // this group's part of the item: the 4 lanes of a row by shuffles (l),
      // then the 4 warps through shared memory
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
      if (gq < G) {
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) {
          red_o[(gw * G + gq) * kHead + nd * 8 + 2 * tq] = oacc[nd][0];
          red_o[(gw * G + gq) * kHead + nd * 8 + 2 * tq + 1] = oacc[nd][1];
        }
        if (tq == 0) {
          red_m[gw * G + gq] = m_run;
          red_l[gw * G + gq] = l_run;
        }
      }
      bar_group(cg);
      const int n_parts = (item.n_c + kItemChunks - 1) / kItemChunks * kGrp;
      const int pc = item.c0 / kItemChunks * kGrp + cg;
      const bool single = n_parts == 1;
      float* part = partials + ((static_cast<size_t>(s) * kv_heads + g) * max_items * kGrp + pc) * G * kPartialFloats;
      for (int e = gtid; e < G * kHead; e += kGroupThreads) {
        const int hh = e / kHead, d = e % kHead;
        float M = kNone;
#pragma unroll
        for (int wv = 0; wv < 4; ++wv) M = fmaxf(M, red_m[wv * G + hh]);
        float Lsum = 0.f, O = 0.f;
#pragma unroll
        for (int wv = 0; wv < 4; ++wv) {
          const float wgt = red_m[wv * G + hh] == kNone ? 0.f : fast_exp2(red_m[wv * G + hh] - M);
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
        // publish this part (the group's writes, ordered by the barrier, are
        // released by the fence before the ticket); the last part of (s, g) to
        // arrive merges all of them
        bar_group(cg);
        if (gtid == 0) {
          griddep_wait();  // the tickets were zeroed by the plan kernel
          __threadfence();
          *g_last = atomicAdd(&tickets[s * kv_heads + g], 1) == n_parts - 1;
          __threadfence();
        }
        bar_group(cg);
        if (*g_last) {
          // per-head max M of m over the parts, then blocks of part weights
          // 2^(m_c - M) in shared memory (with L = sum l_c 2^(m_c - M)); every
          // output sums its column over the parts with independent loads
          const float* all = partials + (static_cast<size_t>(s) * kv_heads + g) * max_items * kGrp * G * kPartialFloats;
          float* hdr = red_o;                      // [G] M, [G] L (this group's buffers)
          float* wts = hdr + 2 * G;                // [block][G] m_c, then weights
          constexpr int kBlock = kMergeBlock;
          if (gtid < G) hdr[gtid] = kNone;
          for (int c0 = 0; c0 < n_parts; c0 += kBlock) {
            const int nb = min(kBlock, n_parts - c0);
            bar_group(cg);
            for (int e = gtid; e < nb * G; e += kGroupThreads) wts[e] = __ldcg(all + (c0 * G + e) * kPartialFloats);
            bar_group(cg);
            if (gtid < G) {
              float M = hdr[gtid];
              for (int cc = 0; cc < nb; ++cc) M = fmaxf(M, wts[cc * G + gtid]);
              hdr[gtid] = M;
              hdr[G + gtid] = 0.f;
            }
          }
          constexpr int kPer = (G * kHead + kGroupThreads - 1) / kGroupThreads;
          float O[kPer];
#pragma unroll
          for (int k = 0; k < kPer; ++k) O[k] = 0.f;
          for (int c0 = 0; c0 < n_parts; c0 += kBlock) {
            const int nb = min(kBlock, n_parts - c0);
            bar_group(cg);
            for (int e = gtid; e < nb * G; e += kGroupThreads) {
              const float mc = __ldcg(all + (c0 * G + e) * kPartialFloats);
              wts[e] = mc == kNone ? 0.f : fast_exp2(mc - hdr[e % G]);
            }
            bar_group(cg);
            if (gtid < G) {
              float Lsum = hdr[G + gtid];
              for (int cc = 0; cc < nb; ++cc)
                Lsum = fmaf(__ldcg(all + ((c0 + cc) * G + gtid) * kPartialFloats + 1), wts[cc * G + gtid], Lsum);
              hdr[G + gtid] = Lsum;
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
              const int e = gtid + k * kGroupThreads;
              if (e < G * kHead) {
                const int hh = e / kHead, d = e % kHead;
                float acc = O[k];
#pragma unroll 4
                for (int cc = 0; cc < nb; ++cc)
                  acc = fmaf(__ldcg(all + ((c0 + cc) * G + hh) * kPartialFloats + 2 + d), wts[cc * G + hh], acc);
                O[k] = acc;
              }
            }
          }
          bar_group(cg);
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int e = gtid + k * kGroupThreads;
            if (e < G * kHead) {
              const int hh = e / kHead, d = e % kHead;
              out[static_cast<size_t>(s) * heads * kHead + (g * G + hh) * kHead + d] = __float2bfloat16_rn(O[k] / hdr[G + hh]);
            }
          }
        }
      }
      bar_group(cg);  // this group's buffers are reused by its next item
      PHASE(1);
    }
    PHASE_FLUSH(g_kime_dec_phase, 8, tid == 0);
  }
  __syncthreads();
#ifdef KIME_PHASE_PROFILE
  if (tid == 0 && blockIdx.x < 1024) g_kime_dec_span[2 * blockIdx.x + 1] = globaltimer();
#endif
}

template <int G, bool kAppend>
cudaError_t launch_decode_g(const CUtensorMap* k_map, const CUtensorMap* v_map, const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                            float scale, const float* cos_t, const float* sin_t, int rope_len, void* k_cache,
                            void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st) {
  static int configured[64] = {0};
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  constexpr uint32_t smem = DecLayout<G>::bytes;
  static_assert(smem <= 232448, "decode shared memory");
  if (dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<G, kAppend>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const int max_items = dec_items_for(cap);
  char* w = static_cast<char*>(ws);
  DecPlan* plan = reinterpret_cast<DecPlan*>(w);
  int32_t* tickets = reinterpret_cast<int32_t*>(w + sizeof(DecPlan));
  int4* items = reinterpret_cast<int4*>(w + dec_ws_items_offset(n_seqs, kv_heads));
  float* partials = reinterpret_cast<float*>(w + dec_ws_head_bytes(n_seqs, kv_heads, cap));
  const long long n_max = static_cast<long long>(max_items) * n_seqs * kv_heads;
  const int grid = static_cast<int>(std::min<long long>(static_cast<long long>(DecCfg<G>::ctas_per_sm) * sms, n_max));
  const int n_static = std::min(grid, n_seqs * kv_heads);
  decode_plan_kernel<<<1, 1024, 0, st>>>(pos, n_seqs, kv_heads, cap, rope_len, n_static, plan, tickets, items,
                                         dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // launched with programmatic stream serialization: its prologue overlaps
  // the plan kernel, whose list it waits for (griddep_wait) before reading it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(DecCfg<G>::threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<G, kAppend>, *k_map, *v_map, static_cast<const uint16_t*>(qkv_new),
                            pos, n_seqs, heads, kv_heads, cap, scale * 1.4426950408889634f, cos_t, sin_t, rope_len,
                            static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
                            static_cast<__nv_bfloat16*>(out), partials, tickets, plan,
                            static_cast<const int4*>(items), max_items, n_static, dev_status);
  return cudaGetLastError();
}

}  // namespace

#ifdef KIME_PHASE_PROFILE
extern "C" int kime_debug_dec_phase_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_kime_dec_phase, sizeof(g_kime_dec_phase));
}
extern "C" int kime_debug_dec_span_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_kime_dec_span, sizeof(g_kime_dec_span));
}
extern "C" int kime_debug_dec_phase_clear() {
  unsigned long long z[16] = {0};
  return cudaMemcpyToSymbol(g_kime_dec_phase, z, sizeof(z));
}
#endif

size_t decode_workspace_bytes(int n_seqs, int heads, int kv_heads, int cap) {
  const int G = heads / kv_heads;
  const size_t parts = static_cast<size_t>(n_seqs) * kv_heads * dec_items_for(cap) * dec_groups_for(G) * G *
                       kPartialFloats * sizeof(float);
  return dec_ws_head_bytes(n_seqs, kv_heads, cap) + parts;
}

cudaError_t launch_kv_append(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                             const float* cos_t, const float* sin_t, int rope_len, void* k_cache, void* v_cache,
                             int32_t* dev_status, cudaStream_t st) {
  kv_append_kernel<<<n_seqs, kAppendThreads, 0, st>>>(static_cast<const uint16_t*>(qkv_new), pos, heads, kv_heads,
                                                      cap, cos_t, sin_t, rope_len, static_cast<uint16_t*>(k_cache),
                                                      static_cast<uint16_t*>(v_cache), dev_status);
  return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap* k_map, const CUtensorMap* v_map, const void* qkv_new, const int32_t* pos,
                          int n_seqs, int heads, int kv_heads, int cap,
                          float scale, const float* cos_t, const float* sin_t, int rope_len, const void* k_cache,
                          const void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st,
                          bool append) {
  void* kc = const_cast<void*>(k_cache);
  void* vc = const_cast<void*>(v_cache);
  switch (heads / kv_heads) {
#define KIME_G(N)                                                                                                    \
  case N:                                                                                                            \
    return append ? launch_decode_g<N, true>(k_map, v_map, qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t,        \
                                             rope_len, kc, vc, out, ws, dev_status, st)                              \
                  : launch_decode_g<N, false>(k_map, v_map, qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t,       \
                                              rope_len, kc, vc, out, ws, dev_status, st);
    KIME_G(1) KIME_G(2) KIME_G(3) KIME_G(4) KIME_G(5) KIME_G(6) KIME_G(7) KIME_G(8)
#undef KIME_G
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kime
