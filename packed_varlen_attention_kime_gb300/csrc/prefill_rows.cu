// prefill_rows.cu -- packed variable-length attention on the sm_103a tensor
// cores over prepared qkv rows (prep.cu: queries rotated and multiplied by
// scale * log2(e), keys rotated, both rounded once to f16, values widened to
// f16, all in the qkv layout).  This is the kernel of kime_attn_varlen for
// BF16 qkv when the workspace holds the prepared rows, and of the chunked
// prefill (kime_attn_chunk) when it holds the chunk's prepared query rows and
// the cache rows widened to f16 (chunk.cu: chunk_prep_kernel).
//
// Semantics (per sequence s, head h, local query i of a length-L sequence):
// out = softmax over visible keys j of scale * <rope(q_i, i), rope(k_j, j)>,
// times v_j.  q is head h of the row; k, v are kv head h / (heads/kv_heads)
// (ffai-argus 0.7.3 src/text.rs, TextTower::block GQA fold).  Key j is
// visible when j < L, j <= i if causal, |i - j| <= window if window >= 0
// (kime-cuda 0.0.3 src/plan.rs, Op::Attention: window None = -1).  For a
// chunk the query row i of sequence s sits at position pos[s] + i and sees
// cache keys 0..pos[s] + i (ffai-argus src/text.rs, CausalSoftmax with offset
// index_pos).  Masked keys
// are left out of the row maximum and get probability zero; no -inf is
// formed (ffai-argus src/text.rs, module doc and CausalSoftmax: deleting the
// mask is bit-identical to adding -inf).
//
// CTA = 640 threads, persistent over units; a unit is two consecutive 128-row
// query tiles A and B of one sequence and one head, which share every K/V
// tile:
//   warpgroups 0, 1  softmax of tile A: warpgroup c takes key columns
//                    64c .. 64c + 63 of every key tile, for all 128 rows
//   warpgroups 2, 3  the same for tile B
//   warpgroup 4      warp 16: TMA producer (Q tiles of two unit slots, a
//                    4-stage K/V ring); warps 17, 18: one MMA issuer (one
//                    thread) per query tile
// The two warpgroups of a tile exchange their partial row maxima through
// shared memory once per key tile, so each thread works on half a row: twice
// the warps of a one-warpgroup-per-tile softmax to hide the latency of each
// step, half the work each.
//
// TMEM (512 columns): S_A 0..127, S_B 128..255, O_A 256..319, O_B 320..383,
// P_A 384..447, P_B 448..511 (f16 P, two keys per 32-bit column).  Per key
// tile t the tile's issuer computes S(t) = Q K^T (M=128, N=128, f16 in, f32
// accumulate); the tile's S buffer takes S(t+1) as soon as both softmax
// warpgroups have loaded their halves of S(t) into registers, so the next S
// is computed while the softmax works.  The softmax forms P(t) = 2^(S -
// m_ref), with a reference maximum m_ref that moves only when a row's maximum
// exceeds it by more than 2^8 (then O and the row sums are rescaled), adds the
// rounded f16 probabilities of its 64 keys into its row sum in float32, and
// stores P(t) into TMEM once PV(t-1) has read P(t-1); the issuer then
// computes O += P(t) V(t) (M=128, N=64, A = P from TMEM).  At the end of a
// unit the two warpgroups of a tile add their row sums and each writes its 32
// output columns of the row, O / l.  Every wait is bounded in time; on a
// timeout every role winds down.
#include <type_traits>

#include "kime_common.cuh"

namespace kime {

namespace {

constexpr int kThreads = 640;
constexpr int kStages = 4;
constexpr uint32_t kTile = kBM * kHead * 2;  // 16 KB: 128 rows x 128 B

// Shared memory (offsets from a 1024-byte aligned base).
struct Layout {
  static constexpr uint32_t q = 0;                    // 2 unit slots x 2 query tiles
  static constexpr uint32_t k = q + 4 * kTile;        // K ring
  static constexpr uint32_t v = k + kStages * kTile;  // V ring
  static constexpr uint32_t xch = v + kStages * kTile;  // per tile: partial row maxima [2][2 halves][128] f32
  static constexpr uint32_t xl = xch + 4096;            // per tile: partial row sums [2 halves][128] f32
  static constexpr uint32_t bar = xl + 2048;
  static constexpr uint32_t bytes = bar + 1024 + 1024;  // + alignment slack
  static_assert(bytes <= 232448, "shared memory per CTA");
};

constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kLazy = 8.f;       // the reference max moves when exceeded by more (log2 units)
constexpr uint32_t kIdescS = idesc_f16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 64, 0, 1);

// Registers (setmaxnreg): every warp starts with the launch count, 96 =
// 65536 / 640 rounded down to a multiple of 8; the four softmax warpgroups go
// to 104 and the producer / issuer warpgroup to 64, which sums to 640 x 96.
constexpr uint32_t kLaunchRegs = 96;
constexpr uint32_t kRegsSoftmax = 104, kRegsCtl = 64;
static_assert(4 * kRegsSoftmax + kRegsCtl == 5 * kLaunchRegs, "register split");
static_assert(kLaunchRegs * kThreads <= 65536 && (kLaunchRegs + 8) * kThreads > 65536, "launch register count");
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

// A unit as the producer publishes it: key tiles are keys kbase + 128 t ..
// kbase + 128 t + 127 for t in [kb, ke) (the union of the two query tiles'
// ranges).  With a window the grid starts at the unit's first visible key,
// q0 - window, when its query tiles then visit fewer tiles than on the
// 128-aligned grid (a 128-row query tile with window 64 then sees 2 key
// tiles, not 3); keys below 0 on such a grid are masked, and their rows
// (another sequence's, or the TMA fill before row 0) never reach the output.
// off: the position of the unit's query row 0 (pos[s] for a chunk, else 0).
struct UnitInfo {
  int32_t u, s, qt0, nt, kb, ke, row0, L, kbase, off;
};

struct Shared {
  uint64_t unit_full[2], unit_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2];   // per query tile: its S has been computed
  uint64_t s_read[2];   // per query tile: its S buffer has been loaded (one arrival per warp)
  uint64_t p_full[2];   // per query tile: P stored (and O rescaled), one arrival per warp
  uint64_t pv_full[2];  // per query tile: its PV has completed
  uint64_t drain[2];    // wind-down after an abort: each issuer's last commit
  UnitInfo info[2];
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Shared) <= 1024, "barrier block");

struct Params {
  int heads, kv_heads, window, causal;
  int cap_pad;  // chunks: rows per (sequence, kv head) of the widened cache rows
  __nv_bfloat16* out;
  WsHeader* hdr;
  const Duo* duos;
  int32_t* dev_status;
};

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

// Query tile w's key-tile ranges in a unit, on the unit's (possibly shifted)
// grid; a chunk's queries sit at positions off + row and see keys 0..off + L - 1.
template <int kMode>
__device__ __forceinline__ void unit_ranges(const UnitInfo& inf, int w, int causal, int window, int& kb, int& ke,
                                            int& fb, int& fe) {
  kb = ke = fb = fe = 0;
  if (w < inf.nt) {
    if constexpr (kMode == 3)
      tile_ranges(inf.L, inf.off + inf.L, inf.off, inf.qt0 + w, 1, -1, kb, ke, fb, fe);
    else
      tile_ranges(inf.L, inf.L - inf.kbase, -inf.kbase, inf.qt0 + w, causal, window, kb, ke, fb, fe);
  }
}

// kMode (same bits in every mode):
//   0  long units: the full key tiles (every row sees all their keys) loop
//      over code without column tests, and each thread stores its own output
//      row (extra code costs more than it saves here);
//   1  short sequences: units end every few key tiles and their stores meet
//      in the store queue, so the epilogue transposes each warp's output
//      chunks among groups of four lanes and every store writes 64
//      contiguous bytes of eight rows; one loop tests each tile;
//   2  a window of at most 128: as 1, with every key tile on the partial path
//      (no 128-key tile is then seen whole by every row);
//   3  chunks against the cache: as 0, with the query tiles from rows_map (the
//      chunk's prepared query rows, [total, heads * 64]) and the K/V tiles from
//      kv_map (the widened cache rows: row (s * kv_heads + g) * cap_pad + key,
//      K in columns 0..63, V in 64..127); causal at positions off + row.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_rows_kernel(const __grid_constant__ CUtensorMap rows_map, const __grid_constant__ CUtensorMap kv_map,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + Layout::bar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  const int causal = p.causal, window = p.window;

  if (tid == 0) {
    tma_prefetch_map(&rows_map);
    if constexpr (kMode == 3) tma_prefetch_map(&kv_map);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->unit_full[i], 1);
      mbar_init(&sh->unit_empty[i], 4);  // tile A, tile B, both issuers
      mbar_init(&sh->q_full[i], 1);
      mbar_init(&sh->q_empty[i], 2);     // both issuers
      mbar_init(&sh->s_full[i], 1);
      mbar_init(&sh->s_read[i], 8);
      mbar_init(&sh->p_full[i], 8);
      mbar_init(&sh->pv_full[i], 1);
      mbar_init(&sh->drain[i], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh->kv_full[i], 1);
      mbar_init(&sh->kv_empty[i], 2);  // both issuers
    }
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
    if (mbar_test(bar, parity)) return true;  // (most waits find their phase complete)
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(p.dev_status, ST_TIMEOUT);
    return false;
  };

  if (wg == 4) {
    regs_dec<kRegsCtl>();
    if (warp == 16 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      griddep_wait();  // the schedule and the prepared rows of the kernels before this one
      const int n_units = p.hdr->n_duos * p.heads;
      const int G = p.heads / p.kv_heads;
      uint32_t n = 0, c = 0, nq = 0;  // units taken, K/V tiles and Q pairs issued
      for (;; ++n) {
        const int slot = n & 1;
        if (!wait(&sh->unit_empty[slot], ((n >> 1) & 1) ^ 1)) break;
        // claimed only once its slot is free, so no unit waits behind a busy CTA
        const int u = atomicAdd(&p.hdr->next_duo, 1);
        UnitInfo inf;
        inf.u = u < n_units ? u : -1;
        if (inf.u >= 0) {
          const Duo d = p.duos[u / p.heads];
          inf.s = d.s; inf.qt0 = d.qt0; inf.nt = d.nt; inf.kb = d.kb; inf.ke = d.ke; inf.row0 = d.row0; inf.L = d.L;
          inf.kbase = 0;
          inf.off = kMode == 3 ? d.off : 0;
          if (kMode != 3 && window >= 0) {
            // the grid from the unit's first visible key when that means fewer tile visits
            const int kbase = d.qt0 * kBM - window;
            int kb, ke, fb, fe, kb2 = 0, ke2 = 0, akb, ake, akb2 = 0, ake2 = 0;
            tile_ranges(d.L, d.L - kbase, -kbase, d.qt0, causal, window, kb, ke, fb, fe);
            tile_ranges(d.L, d.qt0, causal, window, akb, ake, fb, fe);
            if (d.nt == 2) {
              tile_ranges(d.L, d.L - kbase, -kbase, d.qt0 + 1, causal, window, kb2, ke2, fb, fe);
              tile_ranges(d.L, d.qt0 + 1, causal, window, akb2, ake2, fb, fe);
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
        if (!wait(&sh->q_empty[slot], ((n >> 1) & 1) ^ 1)) break;
        uint8_t* q = smem + Layout::q + slot * 2 * kTile;
        mbar_arrive_expect_tx(&sh->q_full[slot], inf.nt * kTile);
        tma_load_2d(q, &rows_map, &sh->q_full[slot], h * kHead, inf.row0 + inf.qt0 * kBM);
        if (inf.nt == 2) tma_load_2d(q + kTile, &rows_map, &sh->q_full[slot], h * kHead, inf.row0 + (inf.qt0 + 1) * kBM);
        ++nq;
        const int kx = (p.heads + g) * kHead, vx = (p.heads + p.kv_heads + g) * kHead;
        bool ok = true;
        for (int t = inf.kb; t < inf.ke; ++t, ++c) {
          const int st = c % kStages;
          if (!wait(&sh->kv_empty[st], ((c / kStages) & 1) ^ 1)) { ok = false; break; }
          const int k0 = inf.kbase + t * kBN;  // the tile's first key
          mbar_arrive_expect_tx(&sh->kv_full[st], 2 * kTile);
          if constexpr (kMode == 3) {
            const int kvrow = (inf.s * p.kv_heads + g) * p.cap_pad + k0;  // widened cache row of the tile's key 0
            tma_load_2d(smem + Layout::k + st * kTile, &kv_map, &sh->kv_full[st], 0, kvrow);
            tma_load_2d(smem + Layout::v + st * kTile, &kv_map, &sh->kv_full[st], kHead, kvrow);
          } else {
            tma_load_2d(smem + Layout::k + st * kTile, &rows_map, &sh->kv_full[st], kx, inf.row0 + k0);
            tma_load_2d(smem + Layout::v + st * kTile, &rows_map, &sh->kv_full[st], vx, inf.row0 + k0);
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // every copy this thread issued lands before the CTA releases its
        // shared memory: the last fill of each stage / Q slot
        for (uint32_t st = 0; st < kStages; ++st)
          if (c > st) mbar_wait(&sh->kv_full[st], (((c - 1 - (c - 1 - st) % kStages)) / kStages) & 1);
        for (uint32_t sl = 0; sl < 2; ++sl)
          if (nq > sl) mbar_wait(&sh->q_full[sl], ((nq - 1 - (nq - 1 - sl) % 2) >> 1) & 1);
      }
    } else if ((warp == 17 || warp == 18) && lane == 0) {
      // ---------------------------------------------------------- MMA issuers
      // one per query tile (warp 17: tile A, warp 18: tile B), so neither
      // tile's MMAs wait on the other tile's softmax
      const int w = warp - 17;
      uint32_t n = 0, c = 0, pc = 0, sc = 0;  // units, key tiles, P tiles, S MMAs of this tile
      const uint32_t tS = tmem + kColS + w * 128, tO = tmem + kColO + w * 64, tP = tmem + kColP + w * 64;
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dk0 = sdesc_sw128(sbase + Layout::k, 16, 1024), dv0 = sdesc_sw128(sbase + Layout::v, 0, 1024);
      for (;; ++n) {
        const int slot = n & 1;
        if (!wait(&sh->unit_full[slot], (n >> 1) & 1)) break;
        const UnitInfo inf = sh->info[slot];
        if (inf.u < 0) break;
        int kb, ke, fb, fe;  // this tile's key tiles; none when the unit has no tile B
        unit_ranges<kMode>(inf, w, causal, window, kb, ke, fb, fe);
        const uint32_t aq = sbase + Layout::q + (slot * 2 + w) * kTile;
        bool ok = wait(&sh->q_full[slot], (n >> 1) & 1);
        // S for the key tile that is number cc of the K/V ring: once that
        // tile is in and the softmax warpgroups have loaded the S before it
        // out of the tile's S buffer.  The softmax loads S(t) before it stores
        // P(t), so waiting for that load, then for P(t), in this order loses
        // nothing, and every wait suspends this thread instead of polling
        // (the softmax warps of its scheduler keep the issue slots).
        // descriptors advance by 32 bytes (2 in the address field) per
        // 16-wide k step; the K stages' differ by their offset
        const uint64_t dq = sdesc_sw128(aq, 16, 1024);
        auto issue_s = [&](uint32_t cc) -> bool {
          if (!wait(&sh->kv_full[cc % kStages], (cc / kStages) & 1)) return false;
          if (sc > 0 && !wait(&sh->s_read[w], (sc - 1) & 1)) return false;
          tc_fence_after();
          const uint64_t dk = dk0 + ((cc % kStages) * kTile >> 4);
#pragma unroll
          for (int ks = 0; ks < kHead / 16; ++ks) tc_mma_ss(tS, dq + 2 * ks, dk + 2 * ks, kIdescS, ks > 0);
          tc_commit(&sh->s_full[w]);
          ++sc;
          return true;
        };
        auto issue_pv = [&](int t, int st) -> bool {
          if (!wait(&sh->p_full[w], pc & 1)) return false;
          ++pc;
          tc_fence_after();
          const uint64_t dv = dv0 + (st * kTile >> 4);  // 2048 bytes (128) per 16 keys
          const uint32_t acc0 = t > kb ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) tc_mma_ts(tO, tP + ks * 8, dv + 128 * ks, kIdescPV, ks > 0 ? 1u : acc0);
          tc_commit(&sh->pv_full[w]);
          return true;
        };
        // the first S of this tile's range (it may start after the unit's first key tile)
        if (ok && ke > kb) ok = issue_s(c + (kb - inf.kb));
        for (int t = inf.kb; ok && t < inf.ke; ++t, ++c) {
          const int st = c % kStages;
          if (t >= kb && t < ke) {
            if (t + 1 < ke && !(ok = issue_s(c + 1))) break;  // S(t+1)
            if (!(ok = issue_pv(t, st))) break;              // PV(t)
          } else {
            // a key tile this query tile does not see: its release must still
            // follow the fill, or this issuer's arrival could complete the
            // stage's previous phase
            if (!(ok = wait(&sh->kv_full[st], (c / kStages) & 1))) break;
          }
          tc_commit(&sh->kv_empty[st]);  // this issuer's MMAs reading stage st are issued
          if (t + 1 == inf.ke) tc_commit(&sh->q_empty[slot]);  // and its last S of the unit
        }
        if (!ok) break;
        if (inf.kb >= inf.ke) tc_commit(&sh->q_empty[slot]);
        mbar_arrive(&sh->unit_empty[slot]);
      }
      if (*abort_flag) {  // every MMA this thread issued completes before TMEM is freed
        tc_commit(&sh->drain[w]);
        mbar_wait(&sh->drain[w], 0);
      }
    }
    __syncwarp();
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int w = wg >> 1, c = wg & 1;  // query tile, key-column half
    const int r = tid & 127;            // row in the tile = TMEM lane
    const int bar_id = 1 + w;           // the tile's 256 softmax threads
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + kColS + 128 * w + 64 * c + lane_off;
    const uint32_t tO = tmem + kColO + 64 * w + 32 * c + lane_off;
    const uint32_t tP = tmem + kColP + 64 * w + 32 * c + lane_off;
    float* xch = reinterpret_cast<float*>(smem + Layout::xch) + w * 512;  // this tile's [2][2 halves][128]
    float* xl = reinterpret_cast<float*>(smem + Layout::xl) + w * 256;    // this tile's [2 halves][128]
    uint32_t n = 0, sc = 0, pvc = 0, xc = 0;
    for (;; ++n) {
      const int slot = n & 1;
      bool ok = wait(&sh->unit_full[slot], (n >> 1) & 1);
      if (named_bar_or(bar_id, 256, !ok)) break;
      const UnitInfo inf = sh->info[slot];
      named_bar_or(bar_id, 256, false);  // every thread has its copy of the unit
      if (c == 0 && r == 0) mbar_arrive(&sh->unit_empty[slot]);
      if (inf.u < 0) break;
      if (w >= inf.nt) continue;  // no tile B in this unit
      const int h = inf.u % p.heads;
      const int i = (inf.qt0 + w) * kBM + r;
      const bool row_ok = i < inf.L;
      int kb, ke, fb, fe;
      unit_ranges<kMode>(inf, w, causal, window, kb, ke, fb, fe);

      // Online softmax with a lazily moved reference max m_ref: P = 2^(S -
      // m_ref), O (accumulated by the PV MMAs) and the row sum l stay relative
      // to m_ref, which moves -- rescaling O and l -- only when a row's max
      // exceeds it by more than 2^8.  Logits arrive in log2 units.
      float m_ref = kNone, l = 0.f;
      // One key tile of the unit.  For long units full_tag says at compile
      // time whether every row sees all of the tile's keys, so the full tiles
      // [fb, fe) -- the run in the middle of the range, nearly all of them on
      // long full-attention layers -- loop over code without the partial
      // tiles' column tests; short units, which alternate between the two
      // kinds, keep one loop that tests each tile (less code).
      auto tile = [&](const int t, auto full_tag) -> bool {
          ok = wait(&sh->s_full[w], sc & 1) && ok;
          ++sc;
          tc_fence_after();
          uint32_t v[64];
          tmem_ld64_wait(tS, v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->s_read[w]);  // the S buffer may take S(t+1)
          // visible keys of this row in this half form one interval [lo, hi]
          // of column indices 0..63 (only partial tiles test columns)
          bool full;
          if constexpr (std::is_same_v<decltype(full_tag), bool>)
            full = t >= fb && t < fe;
          else
            full = decltype(full_tag)::value;
          int lo = 0, hi = 63;
          if (!full) {
            const int k0 = inf.kbase + t * kBN + 64 * c;  // this half's first key
            if constexpr (kMode == 3) {
              hi = min(63, inf.off + i - k0);  // causal at position off + i (below off + L)
            } else {
              hi = min(63, inf.L - 1 - k0);
              if (causal) hi = min(hi, i - k0);
              if (window >= 0) {
                lo = max(0, max(i - window, 0) - k0);  // (a grid may start below key 0)
                hi = min(hi, i + window - k0);
              }
            }
            if (!row_ok) hi = -1;
            lo = min(lo, 64);
            hi = max(hi, -1);
          }
          // this half's maximum: eight running maxima, two keys per three-input
          // max.  On a partial tile that maximum also covers masked columns, so
          // it only bounds the visible one from above: when it cannot move the
          // reference (the usual case after a row's first tile) neither can the
          // visible one, and either gives the same reference below; otherwise
          // the warp takes the maximum again over the visible columns alone
          // (kNone when there are none), tested against a bit word per 32
          // columns.
          float m8[8];
  #pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
  #pragma unroll
          for (int j = 16; j < 64; j += 2)
            m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          if (!full && __any_sync(0xffffffffu, mx > m_ref + kLazy)) {
            uint32_t vis[2];
  #pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int a = lo - 32 * k, b = hi - 32 * k;  // the interval in this word's bit positions
              const uint32_t upto_b = b < 0 ? 0u : (2u << min(b, 31)) - 1u;
              const uint32_t below_a = a <= 0 ? 0u : (a >= 32 ? ~0u : (1u << a) - 1u);
              vis[k] = upto_b & ~below_a;
            }
  #pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = kNone;
  #pragma unroll
            for (int j = 0; j < 64; ++j)
              if ((vis[j >> 5] >> (j & 31)) & 1u) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(v[j]));
            mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          }
          // the row's maximum over both halves
          float* xb = xch + (xc & 1) * 256;
          ++xc;
          xb[c * 128 + r] = mx;
          if (named_bar_or(bar_id, 256, !ok)) {
            ok = false;
            return false;
          }
          mx = fmaxf(mx, xb[(1 - c) * 128 + r]);
          // move the reference max on the first visible keys, or when it is
          // exceeded by more than kLazy
          float alpha = 1.f;
          if (mx > m_ref + kLazy) {
            if (m_ref != kNone) alpha = fast_exp2(m_ref - mx);
            m_ref = mx;
          }
          // P = 2^(x - m_ref): the differences in float32 pairs, rounded to f16
          // pairs, two exponentials per MUFU operation (P in f16, as the MMA
          // takes it)
          uint64_t mm;
          asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m_ref));
          uint32_t pw[32];
  #pragma unroll
          for (int e = 0; e < 32; ++e) {
            uint64_t xx, d;
            asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "r"(v[2 * e]), "r"(v[2 * e + 1]));
            asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(xx), "l"(mm));
            uint32_t hh;
            asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tcvt.rn.satfinite.f16x2.f32 %0, hi, lo;\n\t}"
                : "=r"(hh)
                : "l"(d));
            asm("ex2.approx.f16x2 %0, %1;" : "=r"(pw[e]) : "r"(hh));
          }
          if (!full) {
            // masked columns: probability zero, from the column indices compared
            // with [lo, hi] as f16 pairs (exact for -1..64; each half of a
            // comparison is 0xFFFF when true)
            const uint32_t lo2 = f16x2_splat(lo), hi2 = f16x2_splat(hi);
  #pragma unroll
            for (int e = 0; e < 32; ++e) {
              const uint32_t cols = f16_bits_small(2 * e) | (f16_bits_small(2 * e + 1) << 16);
              uint32_t ge, le;
              asm("set.ge.u32.f16x2 %0, %1, %2;" : "=r"(ge) : "r"(cols), "r"(lo2));
              asm("set.le.u32.f16x2 %0, %1, %2;" : "=r"(le) : "r"(cols), "r"(hi2));
              pw[e] &= ge & le;
            }
          }
          // the row sum of this half: the f16 probabilities the PV MMA takes,
          // each added in float32.  Long units add each widened pair with one
          // packed float32 addition (the same sums, one instruction fewer per
          // pair; faster there, slower on the short-unit instantiations)
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
          for (int e = 0; e < 32; e += 2) {
            if constexpr (kMode == 0 || kMode == 3) {
              add_f16x2_f32x2(s4[0], s4[1], pw[e]);
              add_f16x2_f32x2(s4[2], s4[3], pw[e + 1]);
            } else {
              add_f16x2_f32(s4[0], s4[1], pw[e]);
              add_f16x2_f32(s4[2], s4[3], pw[e + 1]);
            }
          }
          l = l * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
          // PV(t-1) read P(t-1) and accumulated into O: it completes before
          // P(t) is stored and O is rescaled
          if (t > kb) {
            ok = wait(&sh->pv_full[w], pvc & 1) && ok;
            ++pvc;
            tc_fence_after();
          }
          tmem_st32(tP, pw);
          if (t > kb && __any_sync(0xffffffffu, alpha != 1.f)) {  // this half's 32 output columns
            uint32_t ov[32];
            tmem_ld32(tO, ov);
            tmem_wait_ld();
  #pragma unroll
            for (int d = 0; d < 32; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
            tmem_st32(tO, ov);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->p_full[w]);
        return true;
      };
      bool more = true;
      if constexpr (kMode == 2) {
        for (int t = kb; more && t < ke; ++t) more = tile(t, std::false_type{});
      } else if constexpr (kMode == 1) {
        for (int t = kb; more && t < ke; ++t) more = tile(t, true);
      } else {
        for (int t = kb; more && t < fb; ++t) more = tile(t, std::false_type{});
        for (int t = fb; more && t < fe; ++t) more = tile(t, std::true_type{});
        for (int t = fe; more && t < ke; ++t) more = tile(t, std::false_type{});
      }
      // the tile's 256 threads leave together after a failed wait
      if (named_bar_or(bar_id, 256, !ok)) break;
      if (ke > kb) {
        // epilogue: the two halves' row sums added, and this half's 32
        // output columns of the row, O / l
        ok = wait(&sh->pv_full[w], pvc & 1) && ok;
        ++pvc;
        tc_fence_after();
        uint32_t ov[32];
        tmem_ld32(tO, ov);
        xl[c * 128 + r] = l;
        tmem_wait_ld();
        tc_fence_before();
        if (named_bar_or(bar_id, 256, !ok)) break;
        const float lsum = l + xl[(1 - c) * 128 + r];
        // this half's 32 output columns of the row, O / l, as four 16-byte
        // chunks (a row without visible keys computes garbage and is not
        // stored)
        const float inv = 1.f / lsum;
        uint32_t wv[16];
#pragma unroll
        for (int d = 0; d < 32; d += 2) wv[d >> 1] = pack_bf16x2(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv);
        if constexpr (kMode == 1 || kMode == 2) {
          // Transposed among each group of four lanes (two butterfly steps),
          // so that lane 4g + j holds chunk j of rows 4g .. 4g + 3: each store
          // below then writes 64 contiguous bytes of eight rows rather than
          // 16 bytes of 32 rows.
          const int j4 = lane & 3;
#pragma unroll
          for (int m = 0; m < 2; ++m) {  // the off-diagonal 2x2 blocks trade places
            const int out_at = (j4 & 2) ? m : m + 2;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const uint32_t x = (j4 & 2) ? wv[4 * m + w4] : wv[4 * (m + 2) + w4];
              const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 2);
              if (out_at == m) wv[4 * m + w4] = y; else wv[4 * (m + 2) + w4] = y;
            }
          }
#pragma unroll
          for (int b = 0; b < 2; ++b) {  // each 2x2 block is transposed
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const uint32_t x = (j4 & 1) ? wv[4 * (2 * b) + w4] : wv[4 * (2 * b + 1) + w4];
              const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 1);
              if (j4 & 1) wv[4 * (2 * b) + w4] = y; else wv[4 * (2 * b + 1) + w4] = y;
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int ik = i - lane + (lane & ~3) + k;  // the row whose chunk j4 this lane holds in slot k
            if (ik < inf.L) {
              __nv_bfloat16* dst = p.out + static_cast<size_t>(inf.row0 + ik) * p.heads * kHead + h * kHead + 32 * c;
              *reinterpret_cast<uint4*>(dst + 8 * j4) = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
            }
          }
        } else if (row_ok) {
          __nv_bfloat16* dst = p.out + static_cast<size_t>(inf.row0 + i) * p.heads * kHead + h * kHead + 32 * c;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
        }
        // (the partner reads xl[c] before its next barrier with this thread,
        // the first of the next unit, so xl is free to be written again then)
      }
    }
  }

  // Wind down: after an abort the producer and the issuers have waited
  // (bounded) for their own copies and MMAs in flight; then TMEM is freed.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {
template <int kMode>
cudaError_t launch_rows(const CUtensorMap* rows_map, const CUtensorMap* kv_map, const Params& prm, cudaStream_t st) {
  static int configured[64] = {};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    // the register split above assumes the launch count ptxas gave the kernel
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, prefill_rows_kernel<kMode>)) != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
    if ((e = cudaFuncSetAttribute(prefill_rows_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Layout::bytes)) != cudaSuccess)
      return e;
    if (dev < 64) configured[dev] = 1;
  }
  // launched with programmatic stream serialization: its prologue overlaps
  // the kernels before it, whose results it waits for (griddep_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout::bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_rows_kernel<kMode>, *rows_map, *kv_map, prm);
}
}  // namespace

cudaError_t launch_prefill_rows(const CUtensorMap* rows_map, int heads, int kv_heads, int window, int causal,
                                void* out, void* ws, int max_pairs, int short_seqs, int32_t* dev_status,
                                cudaStream_t st) {
  Params prm;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.window = window;
  prm.causal = causal;
  prm.cap_pad = 0;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.hdr = static_cast<WsHeader*>(ws);
  prm.duos = ws_duos(ws, max_pairs);
  prm.dev_status = dev_status;
  if (window >= 0 && window <= 128) return launch_rows<2>(rows_map, rows_map, prm, st);
  return short_seqs ? launch_rows<1>(rows_map, rows_map, prm, st) : launch_rows<0>(rows_map, rows_map, prm, st);
}

cudaError_t launch_prefill_rows_chunk(const CUtensorMap* q_map, const CUtensorMap* kv_map, int heads, int kv_heads,
                                      int cap_pad, void* out, void* ws, int max_pairs, int32_t* dev_status,
                                      cudaStream_t st) {
  Params prm;
  prm.heads = heads;
  prm.kv_heads = kv_heads;
  prm.window = -1;
  prm.causal = 1;
  prm.cap_pad = cap_pad;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.hdr = static_cast<WsHeader*>(ws);
  prm.duos = ws_duos(ws, max_pairs);
  prm.dev_status = dev_status;
  return launch_rows<3>(q_map, kv_map, prm, st);
}

}  // namespace kime
