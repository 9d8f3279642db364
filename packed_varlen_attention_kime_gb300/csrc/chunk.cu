// chunk.cu -- multi-token KV-cache append for chunked prefill.
//
// ffai-argus 0.7.3 src/text.rs, TextTower::block: a block of seq new tokens at
// index_pos is written into the preallocated cache (KvAppend, which refuses a
// block with pos + seq > cap before writing anything), then attends cache rows
// 0..index_pos+seq with CausalSoftmax offset index_pos.  Here the block of
// sequence s is rows cu[s]..cu[s+1]-1 of a packed qkv buffer; its row i is the
// token at position pos[s] + i: its k heads, rotated there (float32, one
// rounding per operation, then bf16 round-to-nearest-even), and its v heads go
// to cache row pos[s] + i of caches [n_seqs, kv_heads, cap, 64].  The
// attention half is the tensor-core prefill kernel reading its keys and values
// from the cache (prefill_tc.cu, kCache).
//
// One warp per token row; lanes stride over the row's kv heads (rotation
// pairs, then v elements).  A sequence whose block would leave
// [0, min(cap, rope_len)) is reported (KIME_DEV_BAD_POS) and no row of it is
// written.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kRowsPerCta = 4;

__global__ void __launch_bounds__(32 * kRowsPerCta)
    kv_append_varlen_kernel(const uint16_t* __restrict__ qkv, const int32_t* __restrict__ cu,
                            const int32_t* __restrict__ pos, int n_seqs, int total, int heads, int kv_heads, int cap,
                            const float* __restrict__ cos_t, const float* __restrict__ sin_t, int rope_len,
                            uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache, int32_t* dev_status) {
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (blockIdx.x == 0) {  // one report per launch for bad positions (empty sequences included)
    bool bad = false;
    for (int q = threadIdx.x; q < n_seqs; q += blockDim.x) {
      const int off = __ldg(pos + q);
      const long long end = static_cast<long long>(off) + (__ldg(cu + q + 1) - __ldg(cu + q));
      bad |= off < 0 || end > cap || end > rope_len;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) report(dev_status, ST_BAD_POS);
  }
  if (r >= total) return;
  // the sequence owning row r: the largest s with cu[s] <= r
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= r) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo, a = __ldg(cu + s), L = __ldg(cu + s + 1) - a, i = r - a;
  if (i < 0 || i >= L) {  // cu is not a valid prefix sum over [0, total)
    if (lane == 0) report(dev_status, ST_BAD_CU);
    return;
  }
  const int off = __ldg(pos + s);
  const long long end = static_cast<long long>(off) + L;
  if (off < 0 || end > cap || end > rope_len) return;  // reported by block 0
  const int P = off + i;
  const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
  const uint16_t* row = qkv + static_cast<size_t>(r) * W;
  const float* c = cos_t + static_cast<size_t>(P) * kHalf;
  const float* sn = sin_t + static_cast<size_t>(P) * kHalf;
  for (int e = lane; e < kv_heads * kHalf; e += 32) {
    const int g = e / kHalf, t = e % kHalf;
    const uint16_t* xk = row + (heads + g) * kHead;
    const float x0 = __uint_as_float(static_cast<uint32_t>(__ldg(xk + t)) << 16);
    const float x1 = __uint_as_float(static_cast<uint32_t>(__ldg(xk + t + kHalf)) << 16);
    float y0, y1;
    rope_pair(x0, x1, __ldg(c + t), __ldg(sn + t), y0, y1);
    const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
    const uint32_t w = pack_bf16x2(y0, y1);
    k_cache[dst + t] = static_cast<uint16_t>(w & 0xffffu);
    k_cache[dst + t + kHalf] = static_cast<uint16_t>(w >> 16);
  }
  // v heads: 8 bytes per lane per step (rows are 16-byte aligned, heads 128 B)
  const uint2* vsrc = reinterpret_cast<const uint2*>(row + (heads + kv_heads) * kHead);
  for (int e = lane; e < kv_heads * (kHead / 4); e += 32) {
    const int g = e / (kHead / 4), t4 = e % (kHead / 4);
    const size_t dst = ((static_cast<size_t>(s) * kv_heads + g) * cap + P) * kHead;
    reinterpret_cast<uint2*>(v_cache + dst)[t4] = __ldg(vsrc + e);
  }
}

}  // namespace

cudaError_t launch_kv_append_varlen(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total,
                                    int heads, int kv_heads, int cap, const float* cos_t, const float* sin_t,
                                    int rope_len, void* k_cache, void* v_cache, int32_t* dev_status,
                                    cudaStream_t st) {
  const int grid = (total + kRowsPerCta - 1) / kRowsPerCta;
  kv_append_varlen_kernel<<<grid, 32 * kRowsPerCta, 0, st>>>(
      static_cast<const uint16_t*>(qkv), cu, pos, n_seqs, total, heads, kv_heads, cap, cos_t, sin_t, rope_len,
      static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), dev_status);
  return cudaGetLastError();
}

}  // namespace kime
