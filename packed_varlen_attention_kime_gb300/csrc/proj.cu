// proj.cu -- the QKV projection of a packed batch on the sm_103a tensor cores,
// qkv = x W^T, with the attention's row preparation fused into its epilogue.
//
// x is [T, hidden] bf16 (token rows), W is [64 (heads + 2 kv_heads), hidden]
// bf16 -- one fused weight stored [out width, in width], q rows, then k, then
// v (kime-cuda 0.0.3 src/plan.rs, Op::Gemm: weight shape [out.width,
// a.width]; ffai-argus 0.7.3 src/text.rs, Block::q: the [960, 576] fusion of
// q, k and v, q pre-scaled by 1/8 at load).  Each output value is a sum over
// hidden of bf16 products accumulated in FP32 by tcgen05.mma (kind::f16, bf16
// A and B, M = 128 token rows, N = 64 per head, K = 16 per instruction).
//
// Two outputs:
//   prepared rows (the fused producer of the attention kernel over prepared
//     rows): each FP32 accumulator row of a q or k head is rotated at the
//     token's position within its own sequence (rotate-half RoPE with the
//     float32 tables, y_t = fma(x_t, c, -(x_{t+32} s)), y_{t+32} = fma(x_{t+32},
//     c, x_t s)), q heads multiplied by scale * log2(e), and rounded once to
//     f16; v heads are rounded to f16 -- the layout and arithmetic of the row
//     preparation pass (prep.cu), from the FP32 products instead of bf16 qkv,
//     so no bf16 qkv is written or read.  A value beyond the f16 range
//     saturates and sets ST_RANGE.
//   bf16 qkv: the accumulators rounded to bf16, no RoPE (the projection alone).
//
// CTA = 192 threads, persistent over output tiles of 128 token rows x 4 heads
// (the last column tile of a row may hold fewer heads; 4 heads a tile rather
// than 3 load 10% fewer operand bytes per product: the SmolLM2 projection
// 0.0273 against 0.0287 ms):
//   warps 0..3  epilogue: thread r owns row r of the tile (TMEM lane r)
//   warp 4      TMA producer: x and W slabs of 64 hidden columns, 4 stages
//   warp 5      MMA issuer (one thread)
// TMEM holds two accumulators of 256 columns, so the epilogue of one tile
// runs while the MMAs of the next accumulate.  Every wait is bounded in time.
#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kPThreads = 192;
constexpr int kPStages = 4;
constexpr int kNH = 4;                          // heads per column tile
constexpr uint32_t kATile = kBM * 64 * 2;       // 16 KB: 128 token rows x 64 hidden (bf16)
constexpr uint32_t kBTile = kNH * 64 * 64 * 2;  // 32 KB: 256 weight rows x 64 hidden
constexpr uint32_t kStageBytes = kATile + kBTile;
constexpr uint32_t kPBar = kPStages * kStageBytes;
constexpr int kCuSmem = 4096;                     // cu_seqlens entries kept in shared memory
constexpr uint32_t kPCu = kPBar + 256;
constexpr uint32_t kPSmem = kPCu + kCuSmem * 4 + 1024;  // + barriers, cu_seqlens, alignment slack
static_assert(kPSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kAccCols = kNH * 64;          // one accumulator
constexpr uint32_t kPTmemCols = 512;             // two accumulators

struct PShared {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(PShared) <= 256, "barrier block");

struct PParams {
  int T, hidden, heads, kv_heads, n_seqs, rope_len, mode;  // mode 0: prepared rows, 1: bf16 qkv
  float qmul;
  const int32_t* cu;
  const float* cos_t;
  const float* sin_t;
  void* out;
  int32_t* dev_status;
};

__global__ void __launch_bounds__(kPThreads, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                    const PParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PShared* sh = reinterpret_cast<PShared*>(smem + kPBar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_heads = p.heads + 2 * p.kv_heads, W = 64 * n_heads;
  const int n_rt = (p.T + kBM - 1) / kBM, n_ct = (n_heads + kNH - 1) / kNH;
  const int n_tiles = n_rt * n_ct, ksl = p.hidden / 64;

  // the epilogue's binary searches for token positions read cu_seqlens from
  // shared memory when it fits (a global-memory search costs a dependent
  // L2 round trip per step, per row, per tile)
  int32_t* cu_s = reinterpret_cast<int32_t*>(smem + kPCu);
  const bool cu_in_smem = p.mode == 0 && p.n_seqs + 1 <= kCuSmem;
  if (cu_in_smem)
    for (int k = tid; k <= p.n_seqs; k += kPThreads) cu_s[k] = __ldg(p.cu + k);
  if (tid == 0) {
    tma_prefetch_map(&x_map);
    tma_prefetch_map(&w_map);
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh->tmem_base, kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  volatile int32_t* abort_flag = &sh->abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(p.dev_status, ST_TIMEOUT);
    return false;
  };

  if (warp == 4) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer
      uint32_t g = 0;  // slabs issued
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int rt = tile / n_ct, ct = tile % n_ct;
        bool ok = true;
        for (int kk = 0; kk < ksl; ++kk, ++g) {
          const uint32_t st = g % kPStages;
          if (!(ok = wait(&sh->empty[st], ((g / kPStages) & 1) ^ 1))) break;
          uint8_t* a = smem + st * kStageBytes;
          mbar_arrive_expect_tx(&sh->full[st], kStageBytes);  // whole boxes land, rows past the ends zero-filled
          tma_load_2d(a, &x_map, &sh->full[st], kk * 64, rt * kBM);
          tma_load_2d(a + kATile, &w_map, &sh->full[st], kk * 64, ct * kNH * 64);
        }
        if (!ok) break;
      }
      if (*abort_flag)  // the last fill of each stage lands before shared memory is released
        for (uint32_t st = 0; st < kPStages; ++st)
          if (g > st) mbar_wait(&sh->full[st], (((g - 1 - (g - 1 - st) % kPStages)) / kPStages) & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t sbase = smem_u32(smem);
      uint32_t g = 0, i = 0;  // slabs consumed, tiles done
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++i) {
        const int ct = tile % n_ct;
        const int nh = min(kNH, n_heads - ct * kNH);
        const uint32_t idesc = idesc_bf16_f32(128, 64 * nh, 0, 0);
        const uint32_t acc = i & 1, d = tmem + acc * kAccCols;
        // the epilogue has read this accumulator out (two tiles ago)
        if (!(ok = wait(&sh->acc_empty[acc], ((i >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        for (int kk = 0; kk < ksl; ++kk, ++g) {
          const uint32_t st = g % kPStages;
          if (!(ok = wait(&sh->full[st], (g / kPStages) & 1))) break;
          tc_fence_after();
          const uint32_t a = sbase + st * kStageBytes, b = a + kATile;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_ss(d, sdesc_sw128(a + ks * 32, 16, 1024), sdesc_sw128(b + ks * 32, 16, 1024), idesc,
                      (kk > 0 || ks > 0) ? 1u : 0u);
          tc_commit(&sh->empty[st]);  // the slab's stage is free once these MMAs complete
        }
        if (ok) tc_commit(&sh->acc_full[acc]);
      }
      if (!ok) {  // every MMA this thread issued completes before TMEM is freed
        tc_commit(&sh->drain);
        mbar_wait(&sh->drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int r = tid;  // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float big = 0.f;  // largest magnitude rounded to f16 (prepared rows)
    uint32_t i = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
      const int rt = tile / n_ct, ct = tile % n_ct;
      const int nh = min(kNH, n_heads - ct * kNH);
      const int row = rt * kBM + r;
      // the token's position within its own sequence: the largest s with cu[s] <= row
      int pos = -1;
      if (p.mode == 0 && row < p.T) {
        const int32_t* cu = cu_in_smem ? cu_s : p.cu;
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (cu[mid] <= row) lo = mid;
          else hi = mid - 1;
        }
        pos = row - cu[lo];
        if (pos >= p.rope_len) pos = -1;  // a row of no valid sequence: converted without rotation
      }
      // the row's table entries, loaded once for the tile's rotated heads and
      // before the wait, so the loads overlap the tile's MMAs
      float4 ct4[8], st4[8];
      const bool any_rot = p.mode == 0 && pos >= 0 && ct * kNH < p.heads + p.kv_heads;
      if (any_rot) {
        const float4* cr = reinterpret_cast<const float4*>(p.cos_t + static_cast<size_t>(pos) * kHalf);
        const float4* sr = reinterpret_cast<const float4*>(p.sin_t + static_cast<size_t>(pos) * kHalf);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          ct4[q] = __ldg(cr + q);
          st4[q] = __ldg(sr + q);
        }
      }
      const uint32_t acc = i & 1;
      bool ok = wait(&sh->acc_full[acc], (i >> 1) & 1);
      tc_fence_after();
      for (int hh = 0; hh < nh; ++hh) {
        uint32_t v[64];
        tmem_ld64_wait(tmem + acc * kAccCols + hh * 64 + lane_off, v);
        const int gh = ct * kNH + hh;  // head number within the qkv row
        if (!ok || row >= p.T) continue;
        if (p.mode == 1) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * W +
                                                gh * 64);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          continue;
        }
        uint32_t y[32];  // f16 pairs of the prepared head
        const bool rotate = gh < p.heads + p.kv_heads && pos >= 0;
        if (rotate) {
          const float mul = gh < p.heads ? p.qmul : 1.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 c4 = ct4[q], s4 = st4[q];
            const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
            float lo2[4], hi2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = 4 * q + e;
              const float a = __uint_as_float(v[t]), b = __uint_as_float(v[t + 32]);
              lo2[e] = __fmaf_rn(a, cc[e], -__fmul_rn(b, ss[e])) * mul;
              hi2[e] = __fmaf_rn(b, cc[e], __fmul_rn(a, ss[e])) * mul;
            }
            big = fmax3(big, fmax3(fabsf(lo2[0]), fabsf(lo2[1]), fabsf(lo2[2])),
                        fmax3(fabsf(lo2[3]), fmax3(fabsf(hi2[0]), fabsf(hi2[1]), fabsf(hi2[2])), fabsf(hi2[3])));
            y[2 * q] = pack_f16x2(lo2[0], lo2[1]);
            y[2 * q + 1] = pack_f16x2(lo2[2], lo2[3]);
            y[16 + 2 * q] = pack_f16x2(hi2[0], hi2[1]);
            y[16 + 2 * q + 1] = pack_f16x2(hi2[2], hi2[3]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float a = __uint_as_float(v[2 * e]), b = __uint_as_float(v[2 * e + 1]);
            if (pos >= 0) big = fmax3(big, fabsf(a), fabsf(b));
            y[e] = pack_f16x2(a, b);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + static_cast<size_t>(row) * W + gh * 64);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_uint4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
      }
      // this accumulator may take the tile after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
      if (!ok) break;
    }
    if (__any_sync(0xffffffffu, big > kF16Max) && lane == 0) report(p.dev_status, ST_RANGE);
  }

  // Wind down: after an abort the producer and the issuer have waited
  // (bounded) for their own copies and MMAs in flight; then TMEM is freed.
  // The grid ends only after the kernel before it (the scheduler, launched
  // before this one and overlapped with it), so the kernel after it finds
  // both results.
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

}  // namespace

cudaError_t launch_qkv_proj(const CUtensorMap* x_map, const CUtensorMap* w_map, int T, int hidden, int heads,
                            int kv_heads, const int32_t* cu, int n_seqs, float scale, const float* cos_t,
                            const float* sin_t, int rope_len, void* out, int mode, int32_t* dev_status,
                            cudaStream_t st) {
  static int configured[64] = {};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    if ((e = cudaFuncSetAttribute(qkv_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem)) !=
        cudaSuccess)
      return e;
    if (dev < 64) configured[dev] = 1;
  }
  PParams prm;
  prm.T = T;
  prm.hidden = hidden;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.n_seqs = n_seqs;
  prm.rope_len = rope_len;
  prm.mode = mode;
  prm.qmul = scale * 1.4426950408889634f;
  prm.cu = cu;
  prm.cos_t = cos_t;
  prm.sin_t = sin_t;
  prm.out = out;
  prm.dev_status = dev_status;
  const int n_heads = heads + 2 * kv_heads;
  const int tiles = ((T + kBM - 1) / kBM) * ((n_heads + kNH - 1) / kNH);
  // launched with programmatic stream serialization: it runs beside the
  // one-CTA scheduler before it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qkv_proj_kernel, *x_map, *w_map, prm);
}

}  // namespace kime
