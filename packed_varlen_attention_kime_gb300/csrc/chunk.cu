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
// attention half is a tensor-core prefill kernel: with room in the workspace
// it runs over rows prepared once by chunk_prep_kernel below
// (prefill_rows.cu, chunk mode), else it reads its keys and values from the
// cache itself (prefill_tc.cu, kCache).
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

// The rows of the chunk attention over prepared rows.  The last q_blocks
// blocks take the chunk rows, one warp per row: its query heads rotated at
// position pos[s] + i with the float32 tables, y_t = fma(x_t, c, -(x_{t+32}
// s)) and y_{t+32} = fma(x_{t+32}, c, x_t s), times scale * log2(e), each
// rounded once to f16 (the arithmetic of the attention kernels that rotate
// their own tiles); lane q of a round holds 16-byte chunk q of the row's
// queries and swaps it with lane q ^ 4, which holds the other halves of its
// pairs.  The blocks before them (launched first: the larger part of the
// work; SmolLM2 chunk step 0.2509 against 0.255 ms with the query rows first)
// take one 128-key tile of one (sequence, kv head) each: cache rows below
// pos[s] + L widened to f16 (K in columns 0..63, V in 64..127; cached keys
// are rotated already), the rest of the tile zero, so the masked keys
// the attention kernel visits are finite; tiles wholly past pos[s] + L are
// never read and are skipped.  With append set (the chunk step) the rows
// pos[s] .. pos[s] + L - 1 are the chunk's own: taken from its qkv rows, the
// key rotated as kv_append_varlen_kernel rotates it (rope_pair, then bf16),
// written to the cache and widened from there, so the step needs no separate
// append and its cache rows are the same bits.  Sequences with positions
// outside [0, min(cap, rope_len)) are skipped (the scheduler reports them and
// lists none of their tiles).  An operand beyond the f16 range saturates and
// sets KIME_DEV_RANGE.
constexpr int kChunkPrepWarps = 4;
// at most 64 registers a thread, so that eight CTAs (32 warps) share an SM:
// at 104 registers (four CTAs) the widening waited on its loads most of the
// time (SmolLM2 chunk step: 49 us, DRAM 45% busy)
constexpr int kChunkPrepCtasPerSm = 8;

__device__ __forceinline__ float absmax_bf16x8(const uint4& x) {
  return fmax3(fmax3(fabsf(bf16lo(x.x)), fabsf(bf16hi(x.x)), fabsf(bf16lo(x.y))),
               fmax3(fabsf(bf16hi(x.y)), fabsf(bf16lo(x.z)), fabsf(bf16hi(x.z))),
               fmaxf(fabsf(bf16lo(x.w)), fabsf(bf16hi(x.w))));
}

__device__ __forceinline__ uint4 widen_bf16x8(const uint4& x) {
  return make_uint4(pack_f16x2(bf16lo(x.x), bf16hi(x.x)), pack_f16x2(bf16lo(x.y), bf16hi(x.y)),
                    pack_f16x2(bf16lo(x.z), bf16hi(x.z)), pack_f16x2(bf16lo(x.w), bf16hi(x.w)));
}

__global__ void __launch_bounds__(32 * kChunkPrepWarps, kChunkPrepCtasPerSm)
    chunk_prep_kernel(const uint16_t* __restrict__ qkv, const int32_t* __restrict__ cu,
                      const int32_t* __restrict__ pos, int n_seqs, int total, int heads, int kv_heads, int cap,
                      int cap_pad, float qmul, const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                      int rope_len, uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache, int append,
                      uint16_t* __restrict__ q16, uint16_t* __restrict__ kv16, int q_blocks, int32_t* dev_status) {
  // the attention kernel may launch once every CTA of this grid has started;
  // it waits for this grid's results before reading them
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float big = 0.f;  // largest magnitude rounded to f16 by this lane
  const int kv_blocks = static_cast<int>(gridDim.x) - q_blocks;
  if (static_cast<int>(blockIdx.x) >= kv_blocks) {
    const int j = (blockIdx.x - kv_blocks) * kChunkPrepWarps + warp;
    if (j < total) {
      int lo = 0, hi = n_seqs - 1;  // the sequence owning row j: the largest s with cu[s] <= j
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= j) lo = mid;
        else hi = mid - 1;
      }
      const int a0 = __ldg(cu + lo), L = __ldg(cu + lo + 1) - a0, i = j - a0, off = __ldg(pos + lo);
      const long long end = static_cast<long long>(off) + L;
      if (i >= 0 && i < L && off >= 0 && end <= cap && end <= rope_len) {
        const int P = off + i;
        const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
        const uint4* src = reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(j) * W);
        uint4* dst = reinterpret_cast<uint4*>(q16 + static_cast<size_t>(j) * heads * kHead);
        const float* crow = cos_t + static_cast<size_t>(P) * kHalf;
        const float* srow = sin_t + static_cast<size_t>(P) * kHalf;
        const int nq = heads * (kHead / 8);  // 16-byte chunks of the row's queries (a multiple of 8)
        // every chunk of a lane sits at the same place in its head (lane mod 8):
        // its rotation pairs' table entries are the same in every round
        const int a = lane & 7, t0 = (a & 3) * 8;
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(crow + t0));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(crow + t0 + 4));
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(srow + t0));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(srow + t0 + 4));
        const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        for (int qb = 0; qb < nq; qb += 128) {
          uint4 xs[4];  // four rounds' loads before any is used
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int q = qb + 32 * k + lane;
            xs[k] = q < nq ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
          if (qb + 32 * k >= nq) break;  // (uniform over the warp)
          const int q = qb + 32 * k + lane;
          const bool in = q < nq;  // chunks q and q ^ 4 are both in range or both out of it
          const uint4 x = xs[k];
          uint4 y;
          y.x = __shfl_xor_sync(0xffffffffu, x.x, 4);
          y.y = __shfl_xor_sync(0xffffffffu, x.y, 4);
          y.z = __shfl_xor_sync(0xffffffffu, x.z, 4);
          y.w = __shfl_xor_sync(0xffffffffu, x.w, 4);
          if (!in) continue;
          const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = bf16lo(xw[e]), x1 = bf16hi(xw[e]), p0 = bf16lo(yw[e]), p1 = bf16hi(yw[e]);
            float r0, r1;
            if (a < 4) {  // y_t = x_t c - x_{t+32} s
              r0 = __fmaf_rn(x0, cc[2 * e], -__fmul_rn(p0, ss[2 * e]));
              r1 = __fmaf_rn(x1, cc[2 * e + 1], -__fmul_rn(p1, ss[2 * e + 1]));
            } else {      // y_{t+32} = x_{t+32} c + x_t s
              r0 = __fmaf_rn(x0, cc[2 * e], __fmul_rn(p0, ss[2 * e]));
              r1 = __fmaf_rn(x1, cc[2 * e + 1], __fmul_rn(p1, ss[2 * e + 1]));
            }
            big = fmax3(big, fabsf(r0 * qmul), fabsf(r1 * qmul));
            ow[e] = pack_f16x2(r0 * qmul, r1 * qmul);
          }
          dst[q] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          }
        }
      }
    }
  } else {
    const int tiles = cap_pad / kBN;
    const int b = static_cast<int>(blockIdx.x), sg = b / tiles, key0 = (b - sg * tiles) * kBN;
    const int s = sg / kv_heads, g = sg - s * kv_heads;
    const int a0 = __ldg(cu + s), off = __ldg(pos + s), L = __ldg(cu + s + 1) - a0;
    const long long end = static_cast<long long>(off) + L;
    if (off >= 0 && L >= 0 && end <= cap && end <= rope_len && key0 < end) {
      const int Lk = static_cast<int>(end);
      const size_t crow0 = static_cast<size_t>(sg) * cap;      // cache row of key 0
      const size_t wrow0 = static_cast<size_t>(sg) * cap_pad;  // widened row of key 0
      // warp w takes keys key0 + 32 w .. + 31 in two rounds of 16, four keys
      // a step, eight lanes a key (16 bytes of K and of V each); a round's
      // loads all before any of its stores
      const int kr = lane >> 3, ch = lane & 7;
      const size_t W = static_cast<size_t>(kHead) * (heads + 2 * kv_heads);
      for (int half = 0; half < 2; ++half) {
        uint4 kx[4], vx[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int key = key0 + warp * 32 + half * 16 + it * 4 + kr;
          kx[it] = vx[it] = make_uint4(0u, 0u, 0u, 0u);
          if (key < Lk) {
            if (append && key >= off) {  // the chunk's row key - off, as qkv holds it
              const uint16_t* row = qkv + static_cast<size_t>(a0 + key - off) * W;
              kx[it] = __ldg(reinterpret_cast<const uint4*>(row + (heads + g) * kHead) + ch);
              vx[it] = __ldg(reinterpret_cast<const uint4*>(row + (heads + kv_heads + g) * kHead) + ch);
            } else {
              kx[it] = __ldg(reinterpret_cast<const uint4*>(k_cache + (crow0 + key) * kHead) + ch);
              vx[it] = __ldg(reinterpret_cast<const uint4*>(v_cache + (crow0 + key) * kHead) + ch);
            }
          }
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int key = key0 + warp * 32 + half * 16 + it * 4 + kr;
          // the other halves of this lane's rotation pairs: lane ch ^ 4 of its key
          uint4 ky;
          ky.x = __shfl_xor_sync(0xffffffffu, kx[it].x, 4);
          ky.y = __shfl_xor_sync(0xffffffffu, kx[it].y, 4);
          ky.z = __shfl_xor_sync(0xffffffffu, kx[it].z, 4);
          ky.w = __shfl_xor_sync(0xffffffffu, kx[it].w, 4);
          uint4* d = reinterpret_cast<uint4*>(kv16 + (wrow0 + key) * (2 * kHead));
          if (key < Lk) {
            uint4 kb = kx[it];
            if (append && key >= off) {
              // k rotated at position key: pair (t, t + 32), t = 8 (ch mod 4) + e;
              // lanes 0-3 of a key hold the t halves, lanes 4-7 the t + 32 halves
              const int t0 = (ch & 3) * 8;
              const float* crow = cos_t + static_cast<size_t>(key) * kHalf + t0;
              const float* srow = sin_t + static_cast<size_t>(key) * kHalf + t0;
              const uint32_t xw[4] = {kx[it].x, kx[it].y, kx[it].z, kx[it].w};
              const uint32_t yw[4] = {ky.x, ky.y, ky.z, ky.w};
              uint32_t ow[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float r[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                  const float x = h2 ? bf16hi(xw[e]) : bf16lo(xw[e]), y = h2 ? bf16hi(yw[e]) : bf16lo(yw[e]);
                  const float c = __ldg(crow + 2 * e + h2), sn = __ldg(srow + 2 * e + h2);
                  float ya, yb;
                  if (ch < 4) {
                    rope_pair(x, y, c, sn, ya, yb);
                    r[h2] = ya;
                  } else {
                    rope_pair(y, x, c, sn, ya, yb);
                    r[h2] = yb;
                  }
                }
                ow[e] = pack_bf16x2(r[0], r[1]);
              }
              kb = make_uint4(ow[0], ow[1], ow[2], ow[3]);
              reinterpret_cast<uint4*>(k_cache + (crow0 + key) * kHead)[ch] = kb;
              reinterpret_cast<uint4*>(v_cache + (crow0 + key) * kHead)[ch] = vx[it];
            }
            big = fmax3(big, absmax_bf16x8(kb), absmax_bf16x8(vx[it]));
            d[ch] = widen_bf16x8(kb);
            d[8 + ch] = widen_bf16x8(vx[it]);
          } else {
            d[ch] = make_uint4(0u, 0u, 0u, 0u);
            d[8 + ch] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
    }
  }
  if (__any_sync(0xffffffffu, big > kF16Max) && lane == 0) report(dev_status, ST_RANGE);
  // this pass runs beside the scheduler (it reads none of its output); it
  // ends only after the scheduler has, so the attention kernel, which waits
  // for this pass, also finds the scheduler's lists complete
  griddep_wait();
}

}  // namespace

cudaError_t launch_chunk_prep(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total, int heads,
                              int kv_heads, int cap, int cap_pad, float scale, const float* cos_t, const float* sin_t,
                              int rope_len, void* k_cache, void* v_cache, int append, void* q16, void* kv16,
                              int32_t* dev_status, cudaStream_t st) {
  const int q_blocks = (total + kChunkPrepWarps - 1) / kChunkPrepWarps;
  const long long kv_blocks = static_cast<long long>(n_seqs) * kv_heads * (cap_pad / kBN);
  if (q_blocks + kv_blocks >= (1LL << 31)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(q_blocks + kv_blocks));
  cfg.blockDim = dim3(32 * kChunkPrepWarps);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float qmul = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, chunk_prep_kernel, static_cast<const uint16_t*>(qkv), cu, pos, n_seqs, total,
                            heads, kv_heads, cap, cap_pad, qmul, cos_t, sin_t, rope_len,
                            static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), append,
                            static_cast<uint16_t*>(q16), static_cast<uint16_t*>(kv16), q_blocks, dev_status);
}

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
