// schedule.cu -- the device-side work scheduler built from cu_seqlens.
//
// One (sequence s, query tile qt) pair per 128 query rows of each sequence,
// the analogue of kime-cpu's per-batch `blocks` table (kime-cpu 0.0.17
// src/kime_cpu/plan.rs, CpuPlan::run: query blocks (s, q0) stepping through
// cu[s]..cu[s+1]; Step::Attention runs blocks x heads tasks).  For each pair
// it records which key tiles the attention kernels visit and which of those
// are "full" (every query row of the tile sees all 128 keys, so no per-column
// test runs).  It also groups the tiles of a sequence two by two ("duos", the
// unit of the tensor-core kernel).  Both lists are ordered longest-first
// (counting sort on the number of key tiles) so the persistent kernels finish
// the expensive work early.
//
// With per-sequence offsets pos (a chunk of new tokens attending the KV cache
// that already holds them, ffai-argus 0.7.3 src/text.rs, TextTower::block with
// index_pos > 0) row i of sequence s sits at position pos[s] + i and its keys
// are cache rows [0, pos[s] + L); a sequence whose positions would leave
// [0, min(cap, rope_len)) is reported and skipped.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 256;
static_assert(kBuckets % 32 == 0, "buckets per lane");

__device__ __forceinline__ int bucket_of(int kb, int ke) { return kBuckets - 1 - min(ke - kb, kBuckets - 1); }

// The tensor-core kernel's unit: tiles 2qp and 2qp+1 of one sequence; cost =
// S tiles the two compute.
__device__ __forceinline__ Duo make_duo(int s, int qp, int a, int L, int off, int causal, int window, int& cost) {
  Duo d;
  d.s = s;
  d.qt0 = 2 * qp;
  d.nt = (2 * qp + 1) * kBM < L ? 2 : 1;
  d.row0 = a;
  d.L = L;
  d.off = off;
  int kb, ke, fb, fe;
  tile_ranges(L, off + L, off, d.qt0, causal, window, kb, ke, fb, fe);
  d.kb = kb;
  d.ke = ke;
  cost = ke - kb;
  if (d.nt == 2) {
    tile_ranges(L, off + L, off, d.qt0 + 1, causal, window, kb, ke, fb, fe);
    d.kb = min(d.kb, kb);
    d.ke = max(d.ke, ke);
    cost += ke - kb;
  }
  return d;
}

// Status of sequence s (0 when it is scheduled) and its offset.
__device__ __forceinline__ int check_seq(const int32_t* cu, const int32_t* pos, int s, int total, int max_seqlen,
                                         int cap, int rope_len, int& off) {
  const int a = cu[s], b = cu[s + 1];
  off = 0;
  if (a < 0 || b < a || b > total) return ST_BAD_CU;
  if (b - a > max_seqlen) return ST_SEQ_TOO_LONG;
  if (pos) {
    off = pos[s];
    const long long end = static_cast<long long>(off) + (b - a);
    if (off < 0 || end > cap || end > rope_len) return ST_BAD_POS;
  }
  return 0;
}

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ pos, int n_seqs, int total,
                    int max_seqlen, int causal, int window, int cap, int rope_len, WsHeader* hdr,
                    Pair* __restrict__ pairs, int max_pairs, Duo* __restrict__ duos, int max_duos,
                    int32_t* dev_status) {
  __shared__ int hist[2][kBuckets];
  __shared__ int cursor[2][kBuckets];
  __shared__ int s_bad;
  // The attention kernel may start now: it sets itself up (barriers, TMEM,
  // tensor map) and waits for this kernel's lists before reading them.
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < 2 * kBuckets; i += blockDim.x) hist[i / kBuckets][i % kBuckets] = 0;
  if (threadIdx.x == 0) {
    s_bad = 0;
    if (n_seqs > 0 && (cu[0] != 0 || cu[n_seqs] != total)) s_bad = ST_BAD_CU;
  }
  __syncthreads();
  // Work split: one thread per sequence, or -- when sequences are long on
  // average (few sequences of many tiles) -- one warp per sequence with its
  // lanes taking the tiles.
  const bool by_warp = n_seqs > 0 && total / n_seqs > 8 * kBM;
  const int lane = threadIdx.x & 31;
  const int s0 = by_warp ? static_cast<int>(threadIdx.x >> 5) : static_cast<int>(threadIdx.x);
  const int ds = by_warp ? static_cast<int>(blockDim.x >> 5) : static_cast<int>(blockDim.x);
  const int t0 = by_warp ? lane : 0, dt = by_warp ? 32 : 1;
  // Pass 1: validate each sequence and histogram its tiles and duos by cost.
  for (int s = s0; s < n_seqs; s += ds) {
    int off;
    const int bad = check_seq(cu, pos, s, total, max_seqlen, cap, rope_len, off);
    if (bad) {
      if (t0 == 0) atomicOr(&s_bad, bad);
      continue;
    }
    const int a = cu[s], L = cu[s + 1] - a;
    for (int qt = t0; qt * kBM < L; qt += dt) {
      int kb, ke, fb, fe;
      tile_ranges(L, off + L, off, qt, causal, window, kb, ke, fb, fe);
      atomicAdd(&hist[0][bucket_of(kb, ke)], 1);
    }
    for (int qp = t0; 2 * qp * kBM < L; qp += dt) {
      int cost;
      make_duo(s, qp, a, L, off, causal, window, cost);
      atomicAdd(&hist[1][bucket_of(0, cost)], 1);
    }
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    // exclusive prefix sums of the two histograms, one warp each: lane j
    // holds buckets 8j .. 8j+7, a warp scan adds the lanes' totals
    const int k = threadIdx.x >> 5;
    constexpr int kPer = kBuckets / 32;
    int local[kPer], sum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      local[q] = sum;
      sum += hist[k][lane * kPer + q];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const int before = incl - sum;
#pragma unroll
    for (int q = 0; q < kPer; ++q) cursor[k][lane * kPer + q] = before + local[q];
    if (lane == 31) {
      if (k == 0) {
        hdr->n_pairs = min(incl, max_pairs);
        hdr->next_unit = 0;
        if (s_bad) report(dev_status, s_bad);
      } else {
        hdr->n_duos = min(incl, max_duos);
        hdr->next_duo = 0;
      }
    }
  }
  __syncthreads();
  // Pass 2: scatter tiles and duos into cost order (longest first).
  for (int s = s0; s < n_seqs; s += ds) {
    int off;
    if (check_seq(cu, pos, s, total, max_seqlen, cap, rope_len, off)) continue;
    const int a = cu[s], L = cu[s + 1] - a;
    for (int qt = t0; qt * kBM < L; qt += dt) {
      int kb, ke, fb, fe;
      tile_ranges(L, off + L, off, qt, causal, window, kb, ke, fb, fe);
      const int at = atomicAdd(&cursor[0][bucket_of(kb, ke)], 1);
      if (at < max_pairs) pairs[at] = Pair{s, qt, kb, ke, fb, fe, a, L};
    }
    for (int qp = t0; 2 * qp * kBM < L; qp += dt) {
      int cost;
      const Duo d = make_duo(s, qp, a, L, off, causal, window, cost);
      const int at = atomicAdd(&cursor[1][bucket_of(0, cost)], 1);
      if (at < max_duos) duos[at] = d;
    }
  }
}

}  // namespace

cudaError_t launch_schedule(const int32_t* cu, const int32_t* pos, int n_seqs, int total, int max_seqlen,
                            int causal, int window, int cap, int rope_len, void* ws, int max_pairs,
                            int32_t* dev_status, cudaStream_t st) {
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  Pair* pairs = ws_pairs(ws);
  Duo* duos = ws_duos(ws, max_pairs);
  schedule_kernel<<<1, kSchedThreads, 0, st>>>(cu, pos, n_seqs, total, max_seqlen, causal, window, cap, rope_len,
                                               hdr, pairs, max_pairs, duos, max_duos_for(n_seqs, total), dev_status);
  return cudaGetLastError();
}

}  // namespace kime
