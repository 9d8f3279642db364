// prefill_tc.cu -- packed variable-length attention over a BF16 fused qkv
// buffer on the sm_103a tensor cores, with RoPE applied in shared memory:
// the kernel of kime_attn_varlen when the workspace has no room for prepared
// rows (see prefill_rows.cu for the kernel over prepared rows), and of chunked
// prefill against the KV cache.  Warp-specialised, two query tiles per CTA
// sharing every K/V tile, ping-pong between two softmax warpgroups.
//
// Semantics (per sequence s, head h, local query i of a length-L sequence):
// out = softmax over visible keys j of scale * <rope(q_i, i), rope(k_j, j)>,
// times v_j.  q is head h of the row; k, v are kv head h / (heads/kv_heads)
// (ffai-argus 0.7.3 src/text.rs, TextTower::block GQA fold).  RoPE is
// rotate-half with the float32 tables of kime-cuda 0.0.3 src/plan.rs
// (fn rope_tables); positions restart at every sequence (kime-cpu 0.0.17
// src/kime_cpu/plan.rs, Step::Rope).  Key j is visible when j < L, j <= i if
// causal, |i - j| <= window if window >= 0 (kime-cuda Op::Attention: window
// None = -1).  Masked keys are skipped, never written as -inf (ffai-argus
// src/text.rs, module doc and CausalSoftmax).
//
// CTA = 512 threads, one unit = (two consecutive 128-row query tiles A, B of
// one sequence, head h), taken from the device schedule:
//   warpgroup 0  softmax for query tile A (TMEM lanes 0..127)
//   warpgroup 1  softmax for query tile B
//   warpgroup 2  RoPE: rotates the unit's Q tiles (double-buffered per unit)
//                and every K tile in shared memory, converts each V tile;
//                thread r owns row r of a tile
//   warpgroup 3  warp 12: TMA producer (Q tiles, 4-stage K/V ring);
//                warps 13, 14: MMA issuers (one thread each, tcgen05.mma), one
//                per query tile, so neither tile's MMAs wait on the other's
// Registers are rebalanced with setmaxnreg: 168 for the softmax warpgroups,
// 112 for RoPE, 64 for the producer / MMA warpgroup (sum 512 x 128).
// MMA operands are f16 (11-bit significand): q and k are rotated in float32
// and rounded once to f16 (q times scale*log2(e) first, so S arrives in log2
// units), V is widened from bf16 exactly, P is rounded to f16.  Inputs must
// stay inside the f16 range (|value| < 65504; conversions saturate).
// TMEM (512 columns): S_A 0..127, S_B 128..255, O_A 256..319, O_B 320..383,
// P_A 384..447, P_B 448..511 (f16 P, two per 32-bit column).  A tile's S
// buffer is refilled as soon as its softmax warpgroup has loaded S(t) into
// registers, so the issuer issues S(t+1) while the warpgroup still works on
// S(t): a warpgroup goes from one key tile to the next without waiting for
// the tensor pipe, and one warpgroup's softmax overlaps the other's MMAs.
// P(t) goes to the tile's own P columns once PV(t-1), which read P(t-1), has
// completed.  The PV MMAs take P from TMEM
// (A operand) and V from shared memory, and accumulate O in TMEM.  A softmax
// warpgroup reads S(t) once, takes P(t) = 2^(S - m_ref) against a reference
// max that moves only when exceeded by more than 2^8 (then O is rescaled in
// TMEM), and stores P(t) into TMEM.  Keeping P out of shared memory leaves its
// bandwidth to the MMA operands Q, K, V.  Every wait is bounded; on a timeout
// every role winds down.
#include <type_traits>

#include "kime_common.cuh"

#ifdef KIME_PHASE_PROFILE
constexpr int kPhaseSlots = 96;  // role bases 0, 16, 32, 40, 48, 56; at most 12 phases each
__device__ unsigned long long g_kime_phase[kPhaseSlots];
// per CTA (globaltimer): entry, first unit claimed, last claim (none left), exit; units taken
__device__ unsigned long long g_kime_span[5 * 256];
#define SPAN(k, v) \
  if (blockIdx.x < 256) g_kime_span[5 * blockIdx.x + (k)] = (v)
// event timeline of the first CTAs: per logging thread (one per role) its own
// slice of globaltimer stamps and tags (code << 16 | argument), plain stores
constexpr int kEvCtas = 4, kEvRoles = 6, kEvMax = 512;
__device__ unsigned long long g_kime_ev_t[kEvCtas * kEvRoles * kEvMax];
__device__ unsigned int g_kime_ev_tag[kEvCtas * kEvRoles * kEvMax];
__device__ int g_kime_ev_n[kEvCtas * kEvRoles];
#define EV(role, code, arg)                                                                   \
  if (blockIdx.x < kEvCtas) {                                                                 \
    const int base_ = (blockIdx.x * kEvRoles + (role)) * kEvMax;                              \
    if (ev_n < kEvMax) {                                                                      \
      g_kime_ev_t[base_ + ev_n] = globaltimer();                                              \
      g_kime_ev_tag[base_ + ev_n] = ((code) << 16) | ((arg) & 0xffff);                        \
    }                                                                                         \
    ++ev_n;                                                                                   \
    g_kime_ev_n[blockIdx.x * kEvRoles + (role)] = ev_n;                                       \
  }
#define EV_DECL int ev_n = 0
#else
#define SPAN(k, v)
#define EV(role, code, arg)
#define EV_DECL
#endif

namespace kime {

namespace {

constexpr int kThreads = 512;
constexpr int kMaxStages = 4;
constexpr uint32_t kTile = kBM * kHead * 2;  // 16 KB: 128 rows x 128 B
// Shared memory: Q (2 unit slots x 2 tiles), the K/V ring, and when the
// kernel rotates the keys itself a ring of RoPE table tiles (cos and sin rows
// of the 128 key positions of a K tile, 2 x 16 KB): 3 K/V stages + 2 table
// stages then, else 4 K/V stages.
template <bool kTab>
struct Layout {
  static constexpr int stages = kTab ? 3 : 4;
  static constexpr int tab_stages = kTab ? 2 : 0;
  static constexpr uint32_t q = 0;
  static constexpr uint32_t k = q + 4 * kTile;
  static constexpr uint32_t v = k + stages * kTile;
  static constexpr uint32_t tab = v + stages * kTile;
  static constexpr uint32_t bar = tab + tab_stages * 2 * kTile;
  static constexpr uint32_t bytes = bar + 512 + 1024;  // + alignment slack
  static_assert(bytes <= 232448, "shared memory per CTA");
};
constexpr uint32_t kTmemCols = 512;
constexpr float kLazy = 8.f;  // the reference max moves when exceeded by more (log2 units)

constexpr uint32_t kIdescS = idesc_f16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 64, 0, 1);

// kbase: the unit's key tiles are keys kbase + 128 t .. kbase + 128 t + 127
// for t in [kb, ke).  With a window (packed sequences) the grid starts at the
// unit's first visible key, q0 - window, when that means fewer tile visits: a
// 128-row query tile with window 64 then sees 2 key tiles, not the 3 of the
// 128-aligned grid.  For q0 < window the grid starts below key 0; those keys
// are masked, and their rows (another sequence's, or the TMA fill before row
// 0) never reach the output.
struct UnitInfo {
  int32_t u, s, qt0, nt, kb, ke, row0, L, off, kbase;
};

struct Shared {
  uint64_t unit_full[2], unit_empty[2];
  uint64_t q_full[2], q_empty[2], qrot[2];
  uint64_t kv_full[kMaxStages], krot[kMaxStages], kv_empty[kMaxStages];
  uint64_t tab_empty[2];  // a table tile has been read (RoPE done with its K tile)
  uint64_t s_full[2][2];    // per query tile, alternating: S(t) and S(t+1) may both be done
  uint64_t s_read[2];  // the softmax warpgroup has loaded its tile's S (one arrival per warp)
  uint64_t p_full[2], pv_full[2];
  uint64_t drain[2];  // wind-down after an abort: each MMA issuer's last commit
  UnitInfo info[2];
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Shared) <= 512, "barrier block");

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

// Per-warpgroup register counts (setmaxnreg).  Every warp starts with the
// launch count, 65536 / kThreads = 128 (__launch_bounds__(kThreads, 1)); a
// .dec must not raise it and an .inc must not lower it (either is an illegal
// instruction), and the counts of the four warpgroups must sum to 4 x 128.
constexpr uint32_t kLaunchRegs = 65536 / kThreads;
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  static_assert(N <= kLaunchRegs && N % 8 == 0 && N >= 24, "setmaxnreg.dec lowers the count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  static_assert(N >= kLaunchRegs && N % 8 == 0 && N <= 256, "setmaxnreg.inc raises the count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
// softmax warpgroups 168, RoPE warpgroup 112, producer / MMA warpgroup 64
constexpr uint32_t kRegsSoftmax = 168, kRegsRope = 112, kRegsIssue = 64;
static_assert(2 * kRegsSoftmax + kRegsRope + kRegsIssue == 4 * kLaunchRegs, "register split");

// One row's cos/sin table entries (32 + 32 floats), loaded ahead of use.
struct TableRow {
  float4 c[8], s[8];
};
__device__ __forceinline__ void load_table_row(TableRow& t, const float* __restrict__ c, const float* __restrict__ s) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    t.c[k] = __ldg(reinterpret_cast<const float4*>(c) + k);
    t.s[k] = __ldg(reinterpret_cast<const float4*>(s) + k);
  }
}

// Row r's entries from a table tile in shared memory: the cos (or sin) rows of
// 128 positions, 128 bytes each, 128-byte swizzled like the operand tiles.
__device__ __forceinline__ void load_table_row_smem(TableRow& t, const uint8_t* ctile, const uint8_t* stile, int r) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int o = r * 128 + ((k ^ (r & 7)) << 4);
    t.c[k] = *reinterpret_cast<const float4*>(ctile + o);
    t.s[k] = *reinterpret_cast<const float4*>(stile + o);
  }
}

// Row r of a 128-byte-swizzled [128 x 64] tile (16-byte chunk k of row r sits
// at chunk k ^ (r & 7)), bf16 on entry, converted in place to the f16 operand
// the MMAs read.  rope_row: rotate-half RoPE with the row's table entries in
// float32 (y_t = fma(x_t, c, -(x_{t+32} s)), y_{t+32} = fma(x_{t+32}, c,
// x_t s)), times `mul`, rounded once to f16.
// convert_row: the bf16 values widened and rounded to f16.  Both keep in `big`
// the largest magnitude they round (beyond kF16Max it saturates).  zero_row: zeros
// (cache rows past a chunk's keys, whose contents are undefined: a NaN there
// would reach O through a zero probability).
__device__ __forceinline__ void rope_row(uint8_t* tile, int r, const TableRow& tb, float mul, float& big) {
  uint8_t* row = tile + r * 128;
  const int sw = r & 7;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4* plo = reinterpret_cast<uint4*>(row + ((k ^ sw) << 4));
    uint4* phi = reinterpret_cast<uint4*>(row + (((k + 4) ^ sw) << 4));
    const uint4 a = *plo, b = *phi;
    const float4 c0 = tb.c[2 * k], c1 = tb.c[2 * k + 1], s0 = tb.s[2 * k], s1 = tb.s[2 * k + 1];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a0, a1, b0, b1;
      {
        const float xa = bf16lo(aw[e]), xb = bf16lo(bw[e]);
        a0 = __fmaf_rn(xa, cc[2 * e], -__fmul_rn(xb, ss[2 * e]));
        b0 = __fmaf_rn(xb, cc[2 * e], __fmul_rn(xa, ss[2 * e]));
      }
      {
        const float xa = bf16hi(aw[e]), xb = bf16hi(bw[e]);
        a1 = __fmaf_rn(xa, cc[2 * e + 1], -__fmul_rn(xb, ss[2 * e + 1]));
        b1 = __fmaf_rn(xb, cc[2 * e + 1], __fmul_rn(xa, ss[2 * e + 1]));
      }
      big = fmax3(big, fmax3(fabsf(a0 * mul), fabsf(a1 * mul), fabsf(b0 * mul)), fabsf(b1 * mul));
      ya[e] = pack_f16x2(a0 * mul, a1 * mul);
      yb[e] = pack_f16x2(b0 * mul, b1 * mul);
    }
    *plo = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *phi = make_uint4(yb[0], yb[1], yb[2], yb[3]);
  }
}

__device__ __forceinline__ void convert_row(uint8_t* tile, int r, float& big) {
  uint4* row = reinterpret_cast<uint4*>(tile + r * 128);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int k = kk ^ (r & 7);  // neighbouring rows touch different banks
    const uint4 a = row[k];
    big = fmax3(big, fmax3(fabsf(bf16lo(a.x)), fabsf(bf16hi(a.x)), fabsf(bf16lo(a.y))),
                fmax3(fabsf(bf16hi(a.y)), fmax3(fabsf(bf16lo(a.z)), fabsf(bf16hi(a.z)), fabsf(bf16lo(a.w))),
                      fabsf(bf16hi(a.w))));
    row[k] = make_uint4(pack_f16x2(bf16lo(a.x), bf16hi(a.x)), pack_f16x2(bf16lo(a.y), bf16hi(a.y)),
                        pack_f16x2(bf16lo(a.z), bf16hi(a.z)), pack_f16x2(bf16lo(a.w), bf16hi(a.w)));
  }
}

__device__ __forceinline__ void zero_row(uint8_t* tile, int r) {
  uint4* row = reinterpret_cast<uint4*>(tile + r * 128);
#pragma unroll
  for (int k = 0; k < 8; ++k) row[k] = make_uint4(0u, 0u, 0u, 0u);
}

struct Params {
  int heads, kv_heads, cap, window, causal;
  float qmul;  // scale * log2(e), folded into q before its f16 rounding
  const float* cos_t;
  const float* sin_t;
  __nv_bfloat16* out;
  WsHeader* hdr;
  const Duo* duos;
  int32_t* dev_status;
};

// kCache = false: a packed batch; Q, K and V are heads of the qkv rows, Q and
// K rotated here.  kCache = true: chunks attending a KV cache that already
// holds them (rotated keys); K and V tiles come from the cache maps, rows past
// the sequence's keys are zeroed, q rows sit at positions off + i.
// kMode (same bits in every mode):
//   0  long units: each key tile tested for being full (every row sees all
//      its keys), one output row per thread in the epilogue (least code);
//   1  short sequences: units end every few key tiles and their stores crowd
//      the store queue, so the epilogue transposes each warp's output chunks
//      among groups of four lanes (per 64-byte half row) and every store
//      writes 64 contiguous bytes of eight rows;
//   2  a window of at most 128: as 1, and every key tile takes the partial
//      path (a query tile's keys then span tiles no row sees whole, so the
//      full-tile code would only take room in the loop).
template <bool kCache, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qkv_map, const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap cos_map,
                      const __grid_constant__ CUtensorMap sin_map, const Params p) {
  constexpr bool kTab = !kCache;  // keys rotated here, tables staged with each K tile
  using Lay = Layout<kTab>;
  constexpr int kStages = Lay::stages;
  constexpr uint32_t kOffQ = Lay::q, kOffK = Lay::k, kOffV = Lay::v, kOffTab = Lay::tab, kOffBar = Lay::bar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + kOffBar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  const int G = p.heads / p.kv_heads;
  if (tid == 0) SPAN(0, globaltimer());
  const int kCausal = kCache ? 1 : p.causal, kWindow = kCache ? -1 : p.window;  // chunks: causal, no window

  if (tid == 0) {
    tma_prefetch_map(&qkv_map);
    if (kCache) {
      tma_prefetch_map(&k_map);
      tma_prefetch_map(&v_map);
    } else {
      tma_prefetch_map(&cos_map);
      tma_prefetch_map(&sin_map);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->unit_full[i], 1);
      mbar_init(&sh->unit_empty[i], 5);  // softmax A, softmax B, two MMA issuers, RoPE
      mbar_init(&sh->q_full[i], 1);
      mbar_init(&sh->q_empty[i], 2);     // both MMA issuers
      mbar_init(&sh->qrot[i], 1);
      mbar_init(&sh->s_full[i][0], 1);
      mbar_init(&sh->s_full[i][1], 1);
      mbar_init(&sh->p_full[i], 1);
      mbar_init(&sh->pv_full[i], 1);
      mbar_init(&sh->drain[i], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh->kv_full[i], 1);
      mbar_init(&sh->krot[i], 1);
      mbar_init(&sh->kv_empty[i], 2);  // both MMA issuers
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sh->s_read[i], 4);
    for (int i = 0; i < 2; ++i) mbar_init(&sh->tab_empty[i], 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  volatile int32_t* abort_flag = &sh->abort;

  // Bounded wait; a timeout anywhere raises the CTA's abort flag, after which
  // every wait returns false at once and every role leaves its loop.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(p.dev_status, ST_TIMEOUT);
    return false;
  };

  if (wg == 3) {
    regs_dec<kRegsIssue>();
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      griddep_wait();  // the schedule written by the kernel before this one
      const int n_units = p.hdr->n_duos * p.heads;
      uint32_t n = 0, c = 0, nq = 0;  // units taken, K/V tiles and Q pairs issued
      EV_DECL;
      PHASE_DECL(4);
      for (;; ++n) {
        const int slot = n & 1;
        PHASE(3);
        if (!wait(&sh->unit_empty[slot], ((n >> 1) & 1) ^ 1)) break;
        PHASE(0);
        // claimed only once its slot is free, so no unit waits behind a busy CTA
        const int u = atomicAdd(&p.hdr->next_duo, 1);
        EV(0, 0, n);
        if (n == 0) SPAN(1, globaltimer());
        if (u >= n_units) {
          SPAN(2, globaltimer());
          SPAN(4, n);
        }
        UnitInfo inf;
        inf.u = u < n_units ? u : -1;
        if (inf.u >= 0) {
          const Duo d = p.duos[u / p.heads];
          inf.s = d.s; inf.qt0 = d.qt0; inf.nt = d.nt; inf.kb = d.kb; inf.ke = d.ke; inf.row0 = d.row0; inf.L = d.L;
          inf.off = kCache ? d.off : 0;
          inf.kbase = 0;
          if (!kCache && kWindow >= 0) {
            // the unit's key tiles on the grid from its first visible key,
            // q0 - window (the union of its query tiles' ranges there), when
            // its query tiles then visit fewer tiles than on the 128-aligned
            // grid -- never more for q0 > window; for q0 < window the grid
            // starts below key 0 (those keys are masked) and is taken only
            // when it visits strictly fewer
            const int kbase = d.qt0 * kBM - kWindow;
            int kb, ke, fb, fe, kb2 = 0, ke2 = 0, akb, ake, akb2 = 0, ake2 = 0;
            tile_ranges(d.L, d.L - kbase, -kbase, d.qt0, kCausal, kWindow, kb, ke, fb, fe);
            tile_ranges(d.L, d.qt0, kCausal, kWindow, akb, ake, fb, fe);
            if (d.nt == 2) {
              tile_ranges(d.L, d.L - kbase, -kbase, d.qt0 + 1, kCausal, kWindow, kb2, ke2, fb, fe);
              tile_ranges(d.L, d.qt0 + 1, kCausal, kWindow, akb2, ake2, fb, fe);
            }
            const int visits = (ke - kb) + (ke2 - kb2), aligned = (ake - akb) + (ake2 - akb2);
            if (kbase > 0 || visits < aligned) {
              inf.kbase = kbase;
              inf.kb = d.nt == 2 ? min(kb, kb2) : kb;
              inf.ke = d.nt == 2 ? max(ke, ke2) : ke;
            }
          }
        }
        sh->info[slot] = inf;
        mbar_arrive(&sh->unit_full[slot]);
        if (inf.u < 0) break;
        const int h = inf.u % p.heads, g = h / G;
        PHASE(3);
        if (!wait(&sh->q_empty[slot], ((n >> 1) & 1) ^ 1)) break;
        PHASE(1);
        uint8_t* q = smem + kOffQ + slot * 2 * kTile;
        mbar_arrive_expect_tx(&sh->q_full[slot], inf.nt * kTile);
        tma_load_2d(q, &qkv_map, &sh->q_full[slot], h * kHead, inf.row0 + inf.qt0 * kBM);
        if (inf.nt == 2)
          tma_load_2d(q + kTile, &qkv_map, &sh->q_full[slot], h * kHead, inf.row0 + (inf.qt0 + 1) * kBM);
        EV(0, 1, n);
        ++nq;
        const int kx = (p.heads + g) * kHead, vx = (p.heads + p.kv_heads + g) * kHead;
        const int kvrow = (inf.s * p.kv_heads + g) * p.cap;  // cache row of key 0
        bool ok = true;
        for (int t = inf.kb; t < inf.ke; ++t, ++c) {
          const int st = c % kStages;
          PHASE(3);
          if (!wait(&sh->kv_empty[st], ((c / kStages) & 1) ^ 1)) { ok = false; break; }
          if (kTab && !wait(&sh->tab_empty[c & 1], ((c >> 1) & 1) ^ 1)) { ok = false; break; }
          PHASE(2);
          EV(0, 2, c);
          mbar_arrive_expect_tx(&sh->kv_full[st], (kTab ? 4 : 2) * kTile);
          if (kCache) {
            tma_load_2d(smem + kOffK + st * kTile, &k_map, &sh->kv_full[st], 0, kvrow + t * kBN);
            tma_load_2d(smem + kOffV + st * kTile, &v_map, &sh->kv_full[st], 0, kvrow + t * kBN);
          } else {
            const int k0 = inf.kbase + t * kBN;  // the tile's first key
            tma_load_2d(smem + kOffK + st * kTile, &qkv_map, &sh->kv_full[st], kx, inf.row0 + k0);
            tma_load_2d(smem + kOffV + st * kTile, &qkv_map, &sh->kv_full[st], vx, inf.row0 + k0);
            if (kTab) {  // the RoPE table rows of key positions k0 .. k0 + 127
              uint8_t* tb = smem + kOffTab + (c & 1) * 2 * kTile;
              tma_load_2d(tb, &cos_map, &sh->kv_full[st], 0, k0);
              tma_load_2d(tb + kTile, &sin_map, &sh->kv_full[st], 0, k0);
            }
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // every copy this thread issued lands before the CTA releases its
        // shared memory: the last fill of each stage / Q slot (earlier fills
        // of a stage completed before the stage was refilled)
        for (uint32_t st = 0; st < kStages; ++st)
          if (c > st) mbar_wait(&sh->kv_full[st], (((c - 1 - (c - 1 - st) % kStages)) / kStages) & 1);
        for (uint32_t sl = 0; sl < 2; ++sl)
          if (nq > sl) mbar_wait(&sh->q_full[sl], ((nq - 1 - (nq - 1 - sl) % 2) >> 1) & 1);
      }
      PHASE_FLUSH(g_kime_phase, 48, true);
    } else if ((warp == 13 || warp == 14) && lane == 0) {
      // ---------------------------------------------------------- MMA issuers
      // one per query tile (warp 13: tile A, warp 14: tile B), so neither
      // tile's PV MMAs queue behind the other tile's softmax
      const int w = warp - 13;
      uint32_t n = 0, c = 0, pc = 0, sc = 0;  // units, key tiles, P tiles, S MMAs of this tile
      EV_DECL;
      const uint32_t tS = tmem + w * 128, tO = tmem + 256 + w * 64, tP = tmem + 384 + w * 64;
      PHASE_DECL(8);
      for (;; ++n) {
        const int slot = n & 1;
        PHASE(4);
        if (!wait(&sh->unit_full[slot], (n >> 1) & 1)) break;
        PHASE(0);
        const UnitInfo inf = sh->info[slot];
        if (inf.u < 0) break;
        const int off = kCache ? inf.off : 0;  // position of the unit's row 0
        int kb = 0, ke = 0, fb, fe;  // this tile's key tiles; none when the unit has no tile B
        if (w < inf.nt)
          tile_ranges(inf.L, off + inf.L - inf.kbase, off - inf.kbase, inf.qt0 + w, kCausal, kWindow, kb, ke, fb, fe);
        const uint32_t aq = smem_u32(smem + kOffQ + slot * 2 * kTile) + w * kTile;
        PHASE(4);
        // the unit's Q, rotated by the RoPE warpgroup
        bool ok = wait(&sh->qrot[slot], (n >> 1) & 1);
        PHASE(1);
        // S for the key tile that is number cc of the K/V ring may be issued
        // once that tile is in (and rotated) and the softmax warpgroup has
        // loaded the S before it out of the tile's S buffer
        // descriptors advance by 32 bytes (2 in the address field) per
        // 16-wide k step; the stages' differ by their offset
        auto s_ready = [&](uint32_t cc) -> bool {
          const uint32_t ph = (cc / kStages) & 1;
          if (!mbar_test(&sh->kv_full[cc % kStages], ph) || !mbar_test(&sh->krot[cc % kStages], ph))
            return false;
          return sc == 0 || mbar_test(&sh->s_read[w], (sc - 1) & 1);
        };
        auto issue_s = [&](int t, uint32_t cc) {
          tc_fence_after();
          const uint64_t dq = sdesc_sw128(aq, 16, 1024);
          const uint64_t dk = sdesc_sw128(smem_u32(smem + kOffK + (cc % kStages) * kTile), 16, 1024);
#pragma unroll
          for (int ks = 0; ks < kHead / 16; ++ks) tc_mma_ss(tS, dq + 2 * ks, dk + 2 * ks, kIdescS, ks > 0);
          tc_commit(&sh->s_full[w][sc & 1]);
          EV(1 + w, 0, t);
          ++sc;
        };
        auto issue_pv = [&](int t, int st) {
          tc_fence_after();
          const uint64_t dv = sdesc_sw128(smem_u32(smem + kOffV + st * kTile), 0, 1024);  // + 128 per 16 keys
          const uint32_t acc0 = t > kb ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) tc_mma_ts(tO, tP + ks * 8, dv + 128 * ks, kIdescPV, ks > 0 ? 1u : acc0);
          tc_commit(&sh->pv_full[w]);
          EV(1 + w, 1, t);
        };
        // Bounded poll: the conditions are tested without blocking, so one
        // thread can wait for whichever of two events comes first.
        uint64_t t0 = 0;
        uint32_t spins = 0;
        auto timed_out = [&]() -> bool {
          if (*abort_flag) return true;
          if ((++spins & 15) != 0) return false;
          const uint64_t now = globaltimer();
          if (t0 == 0) t0 = now;
          if (now - t0 <= kWaitLimitNs) return false;
          *abort_flag = 1;
          report(p.dev_status, ST_TIMEOUT);
          return true;
        };
        // the first S of this tile's range (it may start after the unit's first key tile)
        if (ok && ke > kb) {
          const uint32_t c0 = c + (kb - inf.kb);
          PHASE(4);
          t0 = 0;
          while (ok && !s_ready(c0)) ok = !timed_out();
          PHASE(2);
          if (ok) issue_s(kb, c0);
          PHASE(6);
        }
        for (int t = inf.kb; ok && t < inf.ke; ++t, ++c) {
          const int st = c % kStages;
          if (t >= kb && t < ke) {
            // S(t+1) and PV(t), whichever can go first (S first when both can)
            bool la = t + 1 < ke, pv = true;
            t0 = 0;
            while (la || pv) {
              if (la && s_ready(c + 1)) {
                PHASE(2);
                issue_s(t + 1, c + 1);
                la = false;
                PHASE(6);
              } else if (pv && mbar_try_wait_ns(&sh->p_full[w], pc & 1, la ? 32u : 1000u)) {
                // (suspended while P is pending, briefly when S(t+1) is too,
                // so the poll takes few issue slots from the other warps)
                PHASE(3);
                ++pc;
                issue_pv(t, st);
                pv = false;
                PHASE(5);
              } else if (timed_out()) {
                ok = false;
                break;
              }
            }
            if (!ok) break;
          } else {
            // a key tile this query tile does not see: its release must still
            // follow the fill (and the RoPE pass), or this issuer's arrival
            // could complete the stage's previous phase
            const uint32_t ph = (c / kStages) & 1;
            if (!(ok = wait(&sh->kv_full[st], ph) && wait(&sh->krot[st], ph))) break;
          }
          tc_commit(&sh->kv_empty[st]);  // this issuer's MMAs reading stage st are issued
          if (t + 1 == inf.ke) tc_commit(&sh->q_empty[slot]);  // and its last S of the unit
          PHASE(7);
        }
        if (!ok) break;
        mbar_arrive(&sh->unit_empty[slot]);
      }
      if (*abort_flag) {  // every MMA this thread issued completes before TMEM is freed
        tc_commit(&sh->drain[w]);
        mbar_wait(&sh->drain[w], 0);
      }
      PHASE_FLUSH(g_kime_phase, w == 0 ? 40 : 56, true);
    }
    __syncwarp();
  } else if (wg == 2) {
    regs_dec<kRegsRope>();
    // ------------------------------------------------------------ RoPE
    const int r = tid - 256;  // row of every tile this thread converts
    uint32_t n = 0, c = 0;
    float big = 0.f;  // largest magnitude this thread rounded to f16
    PHASE_DECL(6);
    for (;; ++n) {
      const int slot = n & 1;
      bool ok = wait(&sh->unit_full[slot], (n >> 1) & 1);
      if (named_bar_or(3, 128, !ok)) break;
      PHASE(0);
      const UnitInfo inf = sh->info[slot];
      if (inf.u < 0) break;
      // the unit's query tiles: row r of each, at positions q0 + r
      uint8_t* q = smem + kOffQ + slot * 2 * kTile;
      TableRow tb;
      for (int w = 0; w < inf.nt; ++w) {
        const int i = (inf.qt0 + w) * kBM + r;
        const size_t ti = static_cast<size_t>((kCache ? inf.off : 0) + i) * kHalf;  // table row of position off + i
        if (i < inf.L) load_table_row(tb, p.cos_t + ti, p.sin_t + ti);
        if (w == 0) ok = wait(&sh->q_full[slot], (n >> 1) & 1);
        if (ok) {
          if (i < inf.L)
            rope_row(q + w * kTile, r, tb, p.qmul, big);
          else
            convert_row(q + w * kTile, r, big);
        }
      }
      fence_proxy_async_smem();
      if (named_bar_or(3, 128, !ok)) break;
      PHASE(1);
      if (r == 0) {
        mbar_arrive(&sh->qrot[slot]);
        mbar_arrive(&sh->unit_empty[slot]);  // every thread has its copy of the unit
      }
      const int Lk = (kCache ? inf.off : 0) + inf.L;  // keys of the unit's sequence
      for (int t = inf.kb; t < inf.ke; ++t, ++c) {
        const int st = c % kStages, j = inf.kbase + t * kBN + r;
        PHASE(2);
        ok = wait(&sh->kv_full[st], (c / kStages) & 1);
        PHASE(3);
        if (ok) {
          if (kCache) {  // cached keys are rotated already
            if (j < Lk) {
              convert_row(smem + kOffK + st * kTile, r, big);
              convert_row(smem + kOffV + st * kTile, r, big);
            } else {
              zero_row(smem + kOffK + st * kTile, r);
              zero_row(smem + kOffV + st * kTile, r);
            }
          } else {
            if (j < inf.L) {
              const uint8_t* tab = smem + kOffTab + (c & 1) * 2 * kTile;  // loaded with this K tile
              load_table_row_smem(tb, tab, tab + kTile, r);
              rope_row(smem + kOffK + st * kTile, r, tb, 1.f, big);
            } else {
              convert_row(smem + kOffK + st * kTile, r, big);
            }
            convert_row(smem + kOffV + st * kTile, r, big);
          }
          fence_proxy_async_smem();
        }
        PHASE(4);
        if (named_bar_or(3, 128, !ok)) { ok = false; break; }
        if (r == 0) {
          mbar_arrive(&sh->krot[st]);
          if (kTab) mbar_arrive(&sh->tab_empty[c & 1]);
        }
        PHASE(5);
      }
      if (!ok) break;
    }
    // an operand beyond the f16 range was saturated: reported once per warp
    if (__any_sync(0xffffffffu, big > kF16Max) && lane == 0) report(p.dev_status, ST_RANGE);
    PHASE_FLUSH(g_kime_phase, 32, r == 0);
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warpgroups
    const int w = wg;                  // 0: tile A, 1: tile B
    const int r = tid & 127;           // row in the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + 256 + w * 64 + lane_off, tP = tmem + 384 + w * 64 + lane_off;
    uint32_t n = 0, sc = 0, pvc = 0;
    EV_DECL;
    PHASE_DECL(9);
    for (;; ++n) {
      const int slot = n & 1;
      bool ok = wait(&sh->unit_full[slot], (n >> 1) & 1);
      if (named_bar_or(1 + w, 128, !ok)) break;
      const UnitInfo inf = sh->info[slot];
      named_bar_or(1 + w, 128, false);  // every thread has its copy of the unit
      if (r == 0 && inf.u >= 0) mbar_arrive(&sh->unit_empty[slot]);
      if (inf.u < 0) break;
      const int off = kCache ? inf.off : 0;  // position of the unit's row 0
      if (w >= inf.nt) continue;  // no partner tile in this unit
      const int h = inf.u % p.heads;
      const int qt = inf.qt0 + w, q0 = qt * kBM, i = q0 + r;
      const bool row_ok = i < inf.L;
      int kb, ke, fb, fe;
      tile_ranges(inf.L, off + inf.L - inf.kbase, off - inf.kbase, qt, kCausal, kWindow, kb, ke, fb, fe);
      // chunk rows: the last visible key (this row's position), or none for a padding row
      const int chunk_hi = row_ok ? off + i : -1;

      // Online softmax with a lazily moved reference max: P = 2^(S - m_ref) and
      // O (in TMEM, accumulated by the PV MMAs) stay relative to m_ref, which
      // only moves -- rescaling O and l -- when a row's max exceeds it by more
      // than 2^8.  Logits arrive in log2 units (scale*log2(e) is folded into q).
      float m_ref = kNone, l = 0.f;
      // One key tile; in long units (mode 0) full_tag says at compile time
      // whether every row sees all of the tile's keys, so the full tiles
      // [fb, fe) -- the run in the middle of the range -- loop over code
      // without the partial tiles' column tests.
      auto tile = [&](const int t, auto full_tag) -> bool {
          const int k0 = inf.kbase + t * kBN;
          PHASE(7);
          ok = wait(&sh->s_full[w][sc & 1], (sc >> 1) & 1);
          if (r == 0) EV(3 + w, 0, t);
          ++sc;
          tc_fence_after();
          PHASE(0);
          // the tile's S buffer is free again once every warp has loaded S(t)
          uint32_t v[128];
          tmem_ld128_wait(tmem + w * 128 + lane_off, v);
          tc_fence_before();
          if (lane == 0) mbar_arrive(&sh->s_read[w]);
          PHASE(1);
          // visible keys of this row in this tile form one interval [lo, hi]
          // of column indices (only partial tiles test columns)
          bool full;
          if constexpr (std::is_same_v<decltype(full_tag), bool>)
            full = kMode != 2 && t >= fb && t < fe;
          else
            full = decltype(full_tag)::value;
          int lo = 0, hi = kBN - 1;
          if (!full) {
            if (kCache) {
              hi = min(kBN - 1, chunk_hi - k0);  // causal at position off + i <= off + L - 1
            } else {
              hi = min(kBN - 1, inf.L - 1 - k0);
              if (kCausal) hi = min(hi, i - k0);
              if (kWindow >= 0) {
                lo = max(lo, max(i - kWindow, 0) - k0);  // (a grid may start below key 0)
                hi = min(hi, i + kWindow - k0);
              }
              if (!row_ok) hi = -1;
            }
            lo = min(lo, kBN);
            hi = max(hi, -1);
          }
          // row max: eight running maxima, each taking two keys per three-input
          // max (64 instructions for 128 keys, short dependency chains)
          float m8[8];
  #pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
  #pragma unroll
          for (int j = 16; j < kBN; j += 2)
            m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          // On a partial tile that maximum also covers masked columns, so it only
          // bounds the visible one from above: when it cannot move the reference
          // (the usual case after a row's first tile) the visible maximum cannot
          // either; otherwise the maximum is taken again over the visible
          // columns alone (kNone when there are none), tested against a bit word
          // per 32 columns.
          if (!full && __any_sync(0xffffffffu, mx > m_ref + kLazy)) {
            uint32_t vis[kBN / 32];
  #pragma unroll
            for (int k = 0; k < kBN / 32; ++k) {
              const int a = lo - 32 * k, b = hi - 32 * k;  // the interval in this word's bit positions
              const uint32_t upto_b = b < 0 ? 0u : (2u << min(b, 31)) - 1u;
              const uint32_t below_a = a <= 0 ? 0u : (a >= 32 ? ~0u : (1u << a) - 1u);
              vis[k] = upto_b & ~below_a;
            }
  #pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = kNone;
  #pragma unroll
            for (int j = 0; j < kBN; ++j)
              if ((vis[j >> 5] >> (j & 31)) & 1u) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(v[j]));
            mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          }
          // move the reference max on the first visible keys, or when it is
          // exceeded by more than kLazy (log2 units)
          float alpha = 1.f;
          if (mx > m_ref + kLazy) {
            if (m_ref != kNone) alpha = fast_exp2(m_ref - mx);
            m_ref = mx;
          }
          PHASE(2);
          // P = 2^(x - m_ref): the differences in float32 pairs, rounded to f16
          // pairs (saturating, so no difference becomes infinite), two
          // exponentials per MUFU operation (P in f16, as the MMA takes it).
          // All 64 exponent pairs first (independent chains the schedulers can
          // interleave), then the masked columns set to probability zero.
          uint64_t mm;
          asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m_ref));
          uint32_t pw[64];
  #pragma unroll
          for (int e = 0; e < 64; ++e) {
            uint64_t xx, d;
            asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "r"(v[2 * e]), "r"(v[2 * e + 1]));
            asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(xx), "l"(mm));
            uint32_t h;
            asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tcvt.rn.satfinite.f16x2.f32 %0, hi, lo;\n\t}"
                : "=r"(h)
                : "l"(d));
            asm("ex2.approx.f16x2 %0, %1;" : "=r"(pw[e]) : "r"(h));
          }
          if (!full) {
            // column indices against [lo, hi] as f16 pairs (exact for 0..128):
            // each half of a comparison is 0xFFFF when true
            const uint32_t lo2 = f16x2_splat(lo), hi2 = f16x2_splat(hi);
  #pragma unroll
            for (int e = 0; e < 64; ++e) {
              const uint32_t cols = f16_bits_small(2 * e) | (f16_bits_small(2 * e + 1) << 16);
              uint32_t ge, le;
              asm("set.ge.u32.f16x2 %0, %1, %2;" : "=r"(ge) : "r"(cols), "r"(lo2));
              asm("set.le.u32.f16x2 %0, %1, %2;" : "=r"(le) : "r"(cols), "r"(hi2));
              pw[e] &= ge & le;
            }
          }
          // the row sum: the f16 probabilities the PV MMA takes, each added in
          // float32
          float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  #pragma unroll
          for (int e = 0; e < 64; e += 4) {
            add_f16x2_f32(s8[0], s8[1], pw[e]);
            add_f16x2_f32(s8[2], s8[3], pw[e + 1]);
            add_f16x2_f32(s8[4], s8[5], pw[e + 2]);
            add_f16x2_f32(s8[6], s8[7], pw[e + 3]);
          }
          l = l * alpha + (((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7])));
          // PV(t-1) read P(t-1) from this tile's P columns and accumulated into
          // O: it completes before P(t) is stored and O is rescaled (the
          // exponentials above overlap it)
          if (t > kb) {
            ok = ok && wait(&sh->pv_full[w], (pvc++) & 1);
            tc_fence_after();
          }
          PHASE(3);
  #pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {  // this row's P: keys 2c, 2c+1 in column c
            const uint32_t p8[8] = {pw[8 * q8], pw[8 * q8 + 1], pw[8 * q8 + 2], pw[8 * q8 + 3],
                                    pw[8 * q8 + 4], pw[8 * q8 + 5], pw[8 * q8 + 6], pw[8 * q8 + 7]};
            tmem_st8(tP + q8 * 8, p8);
          }
          PHASE(4);
          if (t > kb && __any_sync(0xffffffffu, alpha != 1.f)) {
            uint32_t ov[64];
            tmem_ld64_wait(tO, ov);
  #pragma unroll
            for (int d = 0; d < kHead; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
            tmem_st64(tO, ov);
          }
          tmem_wait_st();
          PHASE(5);
          tc_fence_before();
          if (named_bar_or(1 + w, 128, !ok)) { ok = false; return false; }
          if (r == 0) mbar_arrive(&sh->p_full[w]);
          if (r == 0) EV(3 + w, 1, t);
          PHASE(6);
        return true;
      };
      bool more = true;
      if constexpr (kMode == 0) {
        for (int t = kb; more && t < fb; ++t) more = tile(t, std::false_type{});
        for (int t = fb; more && t < fe; ++t) more = tile(t, std::true_type{});
        for (int t = fe; more && t < ke; ++t) more = tile(t, std::false_type{});
      } else {
        for (int t = kb; more && t < ke; ++t) more = tile(t, true);
      }
      if (!ok) break;
      ok = wait(&sh->pv_full[w], (pvc++) & 1);
      tc_fence_after();
      uint32_t ov[64];
      tmem_ld64_wait(tO, ov);
      tc_fence_before();
      if (named_bar_or(1 + w, 128, !ok)) break;
      if constexpr (kMode >= 1) {
        // the row's 64 output columns, O / l, as eight 16-byte chunks (a row
        // without visible keys computes garbage and is not stored), then per
        // half row transposed among each group of four lanes (two butterfly
        // steps): lane 4g + j then holds chunk j of the half for rows 4g ..
        // 4g + 3, and each store writes 64 contiguous bytes of eight rows
        const float inv = 1.f / l;
        uint32_t wv[32];
#pragma unroll
        for (int d = 0; d < kHead; d += 2) wv[d >> 1] = pack_bf16x2(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv);
        const int j4 = lane & 3;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t* hv = wv + 16 * hf;
#pragma unroll
          for (int m = 0; m < 2; ++m) {  // the off-diagonal 2x2 blocks trade places
            const int out_at = (j4 & 2) ? m : m + 2;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const uint32_t x = (j4 & 2) ? hv[4 * m + w4] : hv[4 * (m + 2) + w4];
              const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 2);
              if (out_at == m) hv[4 * m + w4] = y; else hv[4 * (m + 2) + w4] = y;
            }
          }
#pragma unroll
          for (int b = 0; b < 2; ++b) {  // each 2x2 block is transposed
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const uint32_t x = (j4 & 1) ? hv[4 * (2 * b) + w4] : hv[4 * (2 * b + 1) + w4];
              const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 1);
              if (j4 & 1) hv[4 * (2 * b) + w4] = y; else hv[4 * (2 * b + 1) + w4] = y;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ik = i - lane + (lane & ~3) + k;  // the row whose chunks j4 this lane holds in slot k
          if (ik < inf.L) {
            __nv_bfloat16* dst = p.out + static_cast<size_t>(inf.row0 + ik) * p.heads * kHead + h * kHead + 8 * j4;
            *reinterpret_cast<uint4*>(dst) = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
            *reinterpret_cast<uint4*>(dst + 32) =
                make_uint4(wv[16 + 4 * k], wv[16 + 4 * k + 1], wv[16 + 4 * k + 2], wv[16 + 4 * k + 3]);
          }
        }
      } else if (row_ok) {
        const float inv = 1.f / l;
        __nv_bfloat16* dst = p.out + static_cast<size_t>(inf.row0 + i) * p.heads * kHead + h * kHead;
#pragma unroll
        for (int d = 0; d < kHead; d += 8) {
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv);
          wv.y = pack_bf16x2(__uint_as_float(ov[d + 2]) * inv, __uint_as_float(ov[d + 3]) * inv);
          wv.z = pack_bf16x2(__uint_as_float(ov[d + 4]) * inv, __uint_as_float(ov[d + 5]) * inv);
          wv.w = pack_bf16x2(__uint_as_float(ov[d + 6]) * inv, __uint_as_float(ov[d + 7]) * inv);
          *reinterpret_cast<uint4*>(dst + d) = wv;
        }
      }
      PHASE(8);
    }
    PHASE_FLUSH(g_kime_phase, 16 * w, r == 0);
  }

  // Wind down: after an abort the producer and the MMA issuers have waited
  // (bounded) for their own copies and MMAs in flight; then TMEM is freed.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) SPAN(3, globaltimer());
}

}  // namespace

#ifdef KIME_PHASE_PROFILE
extern "C" int kime_debug_phase_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_kime_phase, sizeof(g_kime_phase));
}
extern "C" int kime_debug_ev_read(unsigned long long* t, unsigned int* tag, int* n) {  // kEvCtas x kEvRoles slices
  int rc = cudaMemcpyFromSymbol(t, g_kime_ev_t, sizeof(g_kime_ev_t));
  if (!rc) rc = cudaMemcpyFromSymbol(tag, g_kime_ev_tag, sizeof(g_kime_ev_tag));
  if (!rc) rc = cudaMemcpyFromSymbol(n, g_kime_ev_n, sizeof(g_kime_ev_n));
  return rc;
}
extern "C" int kime_debug_ev_clear() {
  int z[kEvCtas * kEvRoles] = {0};
  return cudaMemcpyToSymbol(g_kime_ev_n, z, sizeof(z));
}
extern "C" int kime_debug_span_read(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_kime_span, sizeof(g_kime_span));
}
extern "C" int kime_debug_phase_clear() {
  unsigned long long z[kPhaseSlots] = {0};
  return cudaMemcpyToSymbol(g_kime_phase, z, sizeof(z));
}
#endif

cudaError_t launch_prefill_tc(const CUtensorMap* qkv_map, const CUtensorMap* k_map, const CUtensorMap* v_map,
                              const CUtensorMap* cos_map, const CUtensorMap* sin_map, int heads, int kv_heads, int cap,
                              int window, int causal, float scale, const float* cos_t, const float* sin_t, void* out,
                              void* ws, int max_pairs, int short_units, int32_t* dev_status, cudaStream_t st) {
  // kernel variant: packed sequences (keys rotated here) in one of three
  // modes, or chunks against the caches (long units)
  const bool chunks = k_map != nullptr;
  const int mode = chunks ? 0 : (window >= 0 && window <= 128 ? 2 : (short_units ? 1 : 0));
  static int configured[4][64] = {};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const uint32_t smem_bytes = chunks ? Layout<false>::bytes : Layout<true>::bytes;
  const void* fn = chunks      ? reinterpret_cast<const void*>(prefill_tc_kernel<true, 0>)
                   : mode == 2 ? reinterpret_cast<const void*>(prefill_tc_kernel<false, 2>)
                   : mode == 1 ? reinterpret_cast<const void*>(prefill_tc_kernel<false, 1>)
                               : reinterpret_cast<const void*>(prefill_tc_kernel<false, 0>);
  const int vi = chunks ? 3 : mode;
  if (dev >= 64 || !configured[vi][dev]) {
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) != cudaSuccess)
      return e;
    if (dev < 64) configured[vi][dev] = 1;
  }
  Params prm;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.cap = cap;
  prm.window = window;
  prm.causal = causal;
  prm.qmul = scale * 1.4426950408889634f;
  prm.cos_t = cos_t;
  prm.sin_t = sin_t;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.hdr = static_cast<WsHeader*>(ws);
  prm.duos = ws_duos(ws, max_pairs);
  prm.dev_status = dev_status;
  // launched with programmatic stream serialization: its prologue overlaps the
  // kernel before it (the scheduler), whose lists it waits for (griddep_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (chunks)
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<true, 0>, *qkv_map, *k_map, *v_map, *qkv_map, *qkv_map, prm);
  if (mode == 2)
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<false, 2>, *qkv_map, *qkv_map, *qkv_map, *cos_map, *sin_map,
                              prm);
  if (mode == 1)
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<false, 1>, *qkv_map, *qkv_map, *qkv_map, *cos_map, *sin_map,
                              prm);
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<false, 0>, *qkv_map, *qkv_map, *qkv_map, *cos_map, *sin_map,
                            prm);
}

}  // namespace kime
