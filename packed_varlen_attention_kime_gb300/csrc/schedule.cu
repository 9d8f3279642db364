// schedule.cu -- the device-side work scheduler built from cu_seqlens.
//
// One (sequence s, query tile qt) pair per 128 query rows of each sequence,
// the analogue of kime-cpu's per-batch `blocks` table (kime-cpu 0.0.17
// src/kime_cpu/plan.rs, CpuPlan::run: query blocks (s, q0) stepping through
// cu[s]..cu[s+1]; Step::Attention runs blocks x heads tasks).  For each pair
// it records which key tiles the attention kernels visit and which of those
// are "full" (every query row of the tile sees all 128 keys, so no per-column
// test runs).  Pairs are ordered longest-first (counting sort on the number of
// key tiles) so the persistent kernels finish the expensive work early.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 256;

// ceil(a / b) for a > 0, else 0.
__device__ __forceinline__ int ceil_pos(int a, int b) { return a <= 0 ? 0 : (a + b - 1) / b; }
// Number of key tiles kt >= 0 whose last key kt*128 + 127 is <= x.
__device__ __forceinline__ int tiles_ending_by(int x) { return x < kBN - 1 ? 0 : (x - (kBN - 1)) / kBN + 1; }

// Key-tile ranges of query tile qt of a length-L sequence.
//   visit: k0 < L, causal => k0 <= q1-1, window w => k0 <= q1-1+w and k0+127 >= q0-w
//   full : visit, k0+128 <= L, causal => k0+127 <= q0, window => k0 >= q1-1-w and k0+127 <= q0+w
__device__ __forceinline__ void tile_ranges(int L, int qt, int causal, int window, int& kb, int& ke, int& fb,
                                            int& fe) {
  const int q0 = qt * kBM, q1 = min(q0 + kBM, L);
  kb = 0;
  ke = (L + kBN - 1) / kBN;
  if (causal) ke = min(ke, (q1 - 1) / kBN + 1);
  if (window >= 0) {
    ke = min(ke, (q1 - 1 + window) / kBN + 1);
    kb = max(kb, ceil_pos(q0 - window - (kBN - 1), kBN));
  }
  fb = 0;
  fe = L / kBN;
  if (causal) fe = min(fe, tiles_ending_by(q0));
  if (window >= 0) {
    fe = min(fe, tiles_ending_by(q0 + window));
    fb = max(fb, ceil_pos(q1 - 1 - window, kBN));
  }
  fb = max(fb, kb);
  fe = min(fe, ke);
  if (fe <= fb) fb = fe = kb;
}

__device__ __forceinline__ int bucket_of(int kb, int ke) { return kBuckets - 1 - min(ke - kb, kBuckets - 1); }

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const int32_t* __restrict__ cu, int n_seqs, int total, int max_seqlen, int causal, int window,
                    WsHeader* hdr, Pair* __restrict__ pairs, int max_pairs, int32_t* dev_status) {
  __shared__ int hist[kBuckets];
  __shared__ int cursor[kBuckets];
  __shared__ int s_bad;
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) {
    s_bad = 0;
    if (n_seqs > 0 && (cu[0] != 0 || cu[n_seqs] != total)) s_bad = ST_BAD_CU;
  }
  __syncthreads();
  // Pass 1: validate each sequence and histogram its pairs by cost.
  for (int s = threadIdx.x; s < n_seqs; s += blockDim.x) {
    const int a = cu[s], b = cu[s + 1];
    if (a < 0 || b < a || b > total) {
      atomicOr(&s_bad, ST_BAD_CU);
      continue;
    }
    if (b - a > max_seqlen) {
      atomicOr(&s_bad, ST_SEQ_TOO_LONG);
      continue;
    }
    const int L = b - a;
    for (int qt = 0; qt * kBM < L; ++qt) {
      int kb, ke, fb, fe;
      tile_ranges(L, qt, causal, window, kb, ke, fb, fe);
      atomicAdd(&hist[bucket_of(kb, ke)], 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < kBuckets; ++i) {
      cursor[i] = acc;
      acc += hist[i];
    }
    hdr->n_pairs = min(acc, max_pairs);
    hdr->next_unit = 0;
    if (s_bad) report(dev_status, s_bad);
  }
  __syncthreads();
  // Pass 2: scatter the pairs into cost order (longest first).
  for (int s = threadIdx.x; s < n_seqs; s += blockDim.x) {
    const int a = cu[s], b = cu[s + 1];
    if (a < 0 || b < a || b > total || b - a > max_seqlen) continue;
    const int L = b - a;
    for (int qt = 0; qt * kBM < L; ++qt) {
      int kb, ke, fb, fe;
      tile_ranges(L, qt, causal, window, kb, ke, fb, fe);
      const int at = atomicAdd(&cursor[bucket_of(kb, ke)], 1);
      if (at < max_pairs) pairs[at] = Pair{s, qt, kb, ke, fb, fe, a, L};
    }
  }
}

}  // namespace

cudaError_t launch_schedule(const int32_t* cu, int n_seqs, int total, int max_seqlen, int causal, int window,
                            void* ws, int max_pairs, int32_t* dev_status, cudaStream_t st) {
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  Pair* pairs = reinterpret_cast<Pair*>(static_cast<char*>(ws) + sizeof(WsHeader));
  schedule_kernel<<<1, kSchedThreads, 0, st>>>(cu, n_seqs, total, max_seqlen, causal, window, hdr, pairs,
                                               max_pairs, dev_status);
  return cudaGetLastError();
}

}  // namespace kime
