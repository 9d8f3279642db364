// kime_internal.h -- host-visible internals shared by the translation units of
// libkime_attn (workspace layout, launcher entry points).  Not installed.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kime {

constexpr int kHead = 64;       // head_dim; the library supports exactly this
constexpr int kHalf = 32;       // RoPE pairs per head
constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // keys per tile
constexpr int kDecChunk = 128;  // keys per split-KV decode work item
constexpr int kMaxGroup = 8;    // largest heads/kv_heads the decode path takes

// One (sequence, query tile) of the schedule with its key-tile ranges:
// tiles [kt_begin, kt_end) are visited; [full_begin, full_end) among them need
// no per-column test.  row0 = cu_seqlens[s], L = sequence length.  (For a chunk
// attending the cache the ranges count cache key tiles from position 0.)
struct Pair {
  int32_t s, qt, kt_begin, kt_end, full_begin, full_end, row0, L;
};
static_assert(sizeof(Pair) == 32, "Pair is 32 bytes");

// Two consecutive query tiles (2*qp, 2*qp+1) of one sequence: the unit of the
// tensor-core kernel, whose two softmax warpgroups share each K/V tile.  nt is
// 1 when the sequence's last tile has no partner; [kb, ke) is the union of the
// two tiles' visited key-tile ranges.  off = position of the sequence's first
// query row (0 for a packed sequence, pos[s] for a chunk attending the cache,
// whose keys are then cache rows [0, off + L)).
struct Duo {
  int32_t s, qt0, nt, kb, ke, row0, L, off;
};
static_assert(sizeof(Duo) == 32, "Duo is 32 bytes");

// Head of the prefill workspace.  next_unit / next_duo are the persistent
// kernels' work counters; a unit is (entry, head) = (u / heads, u % heads).
struct WsHeader {
  int32_t next_unit;
  int32_t n_pairs;
  int32_t next_duo;
  int32_t n_duos;
  int32_t pad[12];
};
static_assert(sizeof(WsHeader) == 64, "WsHeader is 64 bytes");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int max_pairs_for(int n_seqs, int total_tokens) { return total_tokens / kBM + n_seqs + 1; }
inline int max_duos_for(int n_seqs, int total_tokens) { return total_tokens / (2 * kBM) + n_seqs + 1; }
inline int dec_chunks_for(int cap) { return (cap + kDecChunk - 1) / kDecChunk; }
constexpr int kDecItemChunks = 16;  // chunks per decode work item
// consumer groups of the decode kernel for G = heads / kv_heads (parts per item)
inline int dec_groups_for(int G) { (void)G; return 1; }
inline int dec_items_for(int cap) { return (dec_chunks_for(cap) + kDecItemChunks - 1) / kDecItemChunks; }
// Decode workspace: a 16-byte plan header (work counter, item count), tickets
// [n_seqs * kv_heads] int32, the work list int4 [n_seqs * kv_heads * items],
// then (256-byte aligned) partials [n_seqs][kv_heads][items][G][68] f32.
inline size_t dec_ws_items_offset(int n_seqs, int kv_heads) {
  return align_up(16 + static_cast<size_t>(n_seqs) * kv_heads * 4, 16);
}
inline size_t dec_ws_head_bytes(int n_seqs, int kv_heads, int cap) {
  return align_up(dec_ws_items_offset(n_seqs, kv_heads) +
                      static_cast<size_t>(n_seqs) * kv_heads * dec_items_for(cap) * 16, 256);
}

// Prefill workspace: header | pairs[max_pairs] | duos[max_duos].
inline size_t varlen_workspace_bytes(int n_seqs, int total_tokens) {
  return sizeof(WsHeader) + static_cast<size_t>(max_pairs_for(n_seqs, total_tokens)) * sizeof(Pair) +
         static_cast<size_t>(max_duos_for(n_seqs, total_tokens)) * sizeof(Duo);
}
inline Pair* ws_pairs(void* ws) { return reinterpret_cast<Pair*>(static_cast<char*>(ws) + sizeof(WsHeader)); }
inline Duo* ws_duos(void* ws, int max_pairs) {
  return reinterpret_cast<Duo*>(static_cast<char*>(ws) + sizeof(WsHeader) + static_cast<size_t>(max_pairs) * sizeof(Pair));
}

size_t decode_workspace_bytes(int n_seqs, int heads, int kv_heads, int cap);
// Records a failing CUDA call's error as the calling thread's
// kime_attn_last_cuda_error() (entry points outside api.cu report through it).
void set_last_cuda_error(int e);

// Launchers (each returns a cudaError_t of the launch).
// pos == nullptr: packed sequences.  Otherwise chunks at offsets pos[s] against
// a cache of cap rows (positions must stay below cap and rope_len).
cudaError_t launch_schedule(const int32_t* cu, const int32_t* pos, int n_seqs, int total, int max_seqlen,
                            int causal, int window, int cap, int rope_len, void* ws, int max_pairs,
                            int32_t* dev_status, cudaStream_t st);
// out_kind: 0 FP32 out, 1 FP16 out, 2 BF16 out (round to nearest even).
cudaError_t launch_varlen_f32(const float* qkv, const int32_t* cu, int n_seqs, int total, int heads, int kv_heads,
                              int window, int causal, float scale, const float* cos_t, const float* sin_t,
                              void* out, int out_kind, void* ws, int max_pairs, int32_t* dev_status,
                              cudaStream_t st);
// The kernel that applies RoPE in shared memory (prefill_tc.cu).  k_map /
// v_map == nullptr: packed sequences, Q and K rotated in the kernel (K with the
// RoPE tables cos_map / sin_map, [rope_len, 32] f32, boxes of 128 rows).
// Otherwise K and V come from caches [n_seqs * kv_heads * cap, 64] (chunks)
// and the table maps are unused.
cudaError_t launch_prefill_tc(const CUtensorMap* qkv_map, const CUtensorMap* k_map, const CUtensorMap* v_map,
                              const CUtensorMap* cos_map, const CUtensorMap* sin_map, int heads, int kv_heads, int cap,
                              int window, int causal, float scale, const float* cos_t, const float* sin_t, void* out,
                              void* ws, int max_pairs, int short_units, int32_t* dev_status, cudaStream_t st);
// (short_units: the sequences are short on average; with a window of at most
// 128 the units are short anyway.  Either selects a kernel whose epilogue
// coalesces its stores.)
// Attention over prepared rows (prefill_rows.cu): rows_map addresses the
// rows written by launch_qkv_prep ([total, W] f16, boxes of 128 rows x 64
// columns, 128-byte swizzle); the work list is the scheduler's in ws.
// short_seqs: the sequences are short on average (units end every few key
// tiles), which selects the kernel whose epilogue coalesces its stores.
cudaError_t launch_prefill_rows(const CUtensorMap* rows_map, int heads, int kv_heads, int window, int causal,
                                void* out, void* ws, int max_pairs, int short_seqs, int32_t* dev_status,
                                cudaStream_t st);
// Chunks attending the cache over prepared rows (prefill_rows.cu, the same
// kernel): q_map addresses the chunk's prepared query rows ([total, heads*64]
// f16), kv_map the widened cache rows ([n_seqs * kv_heads * cap_pad, 128]
// f16: K in columns 0..63, V in 64..127), both with boxes of 128 rows x 64
// columns and 128-byte swizzle; the work list is the chunk scheduler's in ws.
cudaError_t launch_prefill_rows_chunk(const CUtensorMap* q_map, const CUtensorMap* kv_map, int heads, int kv_heads,
                                      int cap_pad, void* out, void* ws, int max_pairs, int32_t* dev_status,
                                      cudaStream_t st);
// The rows launch_prefill_rows_chunk reads (chunk.cu): the chunk's query heads
// rotated at positions pos[s] + i, times scale * log2(e), rounded once to f16
// (q16 [total, heads*64]), and cache rows 0..pos[s] + L_s - 1 of every kv head
// widened to f16 (kv16 as above), zero rows after them to the end of their
// 128-row tile.  append: rows pos[s] .. pos[s] + L_s - 1 come from the chunk's
// qkv rows and are written to the caches too (launch_kv_append_varlen's
// rows, bit for bit), so the chunk step needs no separate append; else the
// caches are only read.  Launched with programmatic stream serialization
// after the scheduler, whose lists it does not read; it ends after the
// scheduler has.
cudaError_t launch_chunk_prep(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total, int heads,
                              int kv_heads, int cap, int cap_pad, float scale, const float* cos_t, const float* sin_t,
                              int rope_len, void* k_cache, void* v_cache, int append, void* q16, void* kv16,
                              int32_t* dev_status, cudaStream_t st);
// The QKV projection qkv = x W^T (proj.cu): x_map over x [T, hidden] bf16
// (boxes of 64 columns x 128 rows), w_map over W [64 (heads + 2 kv_heads),
// hidden] bf16 (boxes of 64 columns x 256 rows), both with 128-byte swizzle;
// hidden a multiple of 64.  mode 0 writes the prepared rows (as
// launch_qkv_prep does from bf16 qkv: RoPE at the positions cu gives, q times
// scale * log2(e), f16), mode 1 the bf16 qkv rows (cu, tables unused).
cudaError_t launch_qkv_proj(const CUtensorMap* x_map, const CUtensorMap* w_map, int T, int hidden, int heads,
                            int kv_heads, const int32_t* cu, int n_seqs, float scale, const float* cos_t,
                            const float* sin_t, int rope_len, void* out, int mode, int32_t* dev_status,
                            cudaStream_t st);
// A packed batch's qkv rows prepared for the attention kernel (prep.cu):
// queries rotated at their positions and scaled by scale * log2(e), keys
// rotated, all rounded to f16, values widened to f16; out [total, W] f16.
// Any of them beyond the f16 range (saturated) sets ST_RANGE in dev_status.
// 3xTF32 FP32 path: after the scheduler, one kernel that reads the FP32 qkv
// rows through qkv_map (f32 [total, W], 32-column x 64-row boxes, 128-byte
// swizzle), rotates, scales, splits and transposes its operands itself and
// writes out [total, heads*64] f32.
cudaError_t launch_prefill_3xtf32(const CUtensorMap* qkv_map, int heads, int kv_heads, int window, int causal,
                                  float scale, const float* cos_t, const float* sin_t, float* out, void* ws,
                                  int32_t* dev_status, cudaStream_t st);
cudaError_t launch_qkv_prep(const void* qkv, const int32_t* cu, int n_seqs, int total, int heads, int kv_heads,
                            float scale, const float* cos_t, const float* sin_t, int rope_len, void* out,
                            int32_t* dev_status, cudaStream_t st);
cudaError_t launch_kv_append_varlen(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total,
                                    int heads, int kv_heads, int cap, const float* cos_t, const float* sin_t,
                                    int rope_len, void* k_cache, void* v_cache, int32_t* dev_status,
                                    cudaStream_t st);
cudaError_t launch_kv_append(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int cap,
                             const float* cos_t, const float* sin_t, int rope_len, void* k_cache, void* v_cache,
                             int32_t* dev_status, cudaStream_t st);
// k_map / v_map: the caches as [n_seqs * kv_heads * cap, 64] bf16 rows (boxes
// of 128 rows, 128-byte swizzle).
cudaError_t launch_decode(const CUtensorMap* k_map, const CUtensorMap* v_map, const void* qkv_new, const int32_t* pos,
                          int n_seqs, int heads, int kv_heads, int cap,
                          float scale, const float* cos_t, const float* sin_t, int rope_len, const void* k_cache,
                          const void* v_cache, void* out, void* ws, int32_t* dev_status, cudaStream_t st,
                          bool append);

}  // namespace kime
