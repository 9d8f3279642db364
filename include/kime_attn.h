/*
 * kime_attn.h -- C ABI of libkime_attn: packed variable-length multi-head
 * attention (head_dim 64) over a fused qkv row buffer, with RoPE applied to q
 * and k on load, for one NVIDIA GB300 (sm_103a).
 *
 * Sources of the semantics (docs.rs pages):
 *   kime-cpu 0.0.17, src/kime_cpu/plan.rs   -- Step::Rope, Step::Attention, CpuPlan::run
 *   kime-cuda 0.0.3, src/plan.rs            -- Op::Attention lowering, fn rope_tables
 *   ffai-argus 0.7.3, src/text.rs           -- CausalSoftmax, KvAppend, TextTower::block
 *
 * Conventions shared by every entry point:
 *  - All tensors are caller-owned and row-major.  Device pointers must be
 *    16-byte aligned.  The library allocates nothing and never synchronises;
 *    all work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) on the current device.
 *  - A host-detectable error returns KIME_EINVAL or KIME_ERANGE and enqueues
 *    nothing.  A failed launch returns KIME_ECUDA.
 *  - Errors found on the device (malformed cu_seqlens, an out-of-range
 *    position, a timed-out wait) OR a KIME_DEV_* bit into *dev_status when
 *    dev_status is non-NULL (device int32, never cleared by the library) and
 *    skip the offending sequence; they never trap.
 *  - head_dim must be 64.  qkv rows are [q heads | k heads | v heads], 64
 *    columns per head, width W = 64*(heads + 2*kv_heads).  q head h reads kv
 *    head h / (heads / kv_heads) (grouped-query attention, ffai-argus
 *    TextTower::block GQA fold).
 *  - RoPE is rotate-half: element t pairs with t+32,
 *      y[t]    = x[t]*cos[p][t]    - x[t+32]*sin[p][t]
 *      y[t+32] = x[t+32]*cos[p][t] + x[t]*sin[p][t],
 *    at the token's position p inside its own sequence (kime-cpu Step::Rope:
 *    the row index minus the start of its sequence).  Tables are float32
 *    [rope_len, 32] device arrays, e.g. from kime_rope_tables().
 */
#ifndef KIME_ATTN_H
#define KIME_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KIME_OK = 0,
  KIME_EINVAL = -1,  /* malformed argument (null pointer, head_dim != 64, heads % kv_heads, ...) */
  KIME_ERANGE = -2,  /* a size out of range (workspace too small, max_seqlen > rope_len, ...) */
  KIME_ECUDA = -3,   /* a CUDA call failed; see kime_attn_last_cuda_error() */
  KIME_ETIMEOUT = -4 /* reserved for callers mapping KIME_DEV_TIMEOUT to a status */
} kime_status;

/* Element types of qkv and out.  KIME_F32_F16OUT / KIME_F32_BF16OUT: FP32 qkv
 * and a 16-bit output, the mixed precision of kime-cuda 0.0.3 src/plan.rs
 * (fn types: with Precision::F16 attention's qkv stays FP32 -- FP16 rounding of
 * q and k would move ModernBERT's softmax -- while its output is FP16).
 * KIME_F32_3XTF32: FP32 qkv and FP32 out, with QK^T and PV on the tensor cores
 * as three TF32 products each (x = hi + lo, hi = x rounded to TF32; a b taken
 * as a_lo b_hi + a_hi b_lo + a_hi b_hi, FP32 accumulate): the FP32 accuracy
 * contract at TF32 tensor rates (kime-cuda's FP32 attention on tensor cores);
 * the workspace of op 0 suffices (op 4 gives the same size). */
typedef enum {
  KIME_F32 = 0,
  KIME_BF16 = 1,
  KIME_F32_F16OUT = 2,
  KIME_F32_BF16OUT = 3,
  KIME_F32_3XTF32 = 4
} kime_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define KIME_DEV_BAD_CU 1       /* cu_seqlens not monotone, outside [0,total], cu[0]!=0 or cu[n]!=total */
#define KIME_DEV_SEQ_TOO_LONG 2 /* a sequence longer than max_seqlen: it is skipped */
#define KIME_DEV_BAD_POS 4      /* a decode/append position outside [0, min(cap, rope_len)): skipped */
#define KIME_DEV_TIMEOUT 8      /* a pipeline wait ran past its time limit; the work item is abandoned */
#define KIME_DEV_RANGE 16       /* BF16 path: a rotated (and scaled) q or k, or a v, beyond the f16 range (|x| > 65504)
                                   was rounded to f16 for the tensor cores and saturated; the results are computed
                                   from the saturated values */

/* kime_attn_varlen -- attention over a packed batch of variable-length
 * sequences (kime-cuda Op::Attention / kime-cpu Step::Attention, with the RoPE
 * step fused into the load).
 *
 * For sequence s with rows cu_seqlens[s] .. cu_seqlens[s+1]-1 (length L), head
 * h, local query i:
 *   out[cu[s]+i, 64h:64h+64] = sum_{j in A(i)} softmax_j(scale * <rope(q_i,i), rope(k_j,j)>) v_j
 * with A(i) = { j < L : (!causal || j <= i) && (window < 0 || |i-j| <= window) }.
 * window = -1 means none (kime-cuda encodes window None as -1); causal with
 * offset 0 is ffai-argus CausalSoftmax.  Masked keys are skipped, never
 * materialised.
 *
 *  qkv          device, [total_tokens, W]: FP32 (KIME_F32, KIME_F32_F16OUT,
 *               KIME_F32_BF16OUT, KIME_F32_3XTF32) or BF16 (KIME_BF16)
 *  cu_seqlens   device int32 [n_seqs+1], cu[0]=0, non-decreasing, cu[n]=total_tokens
 *  max_seqlen   host upper bound on every sequence length; must be <= rope_len
 *  window       -1 or >= 0; causal 0/1; scale > 0 (0.125, or 1 if q is pre-scaled)
 *  rope_cos/sin device float32 [rope_len, 32]
 *  out          device, [total_tokens, heads*64]: FP32 (KIME_F32,
 *               KIME_F32_3XTF32), BF16
 *               (KIME_BF16, KIME_F32_BF16OUT) or FP16 (KIME_F32_F16OUT),
 *               rounded to nearest even from FP32; rows of skipped sequences
 *               are left untouched
 *  workspace    device scratch of at least kime_attn_workspace_bytes(0, ...)
 *               bytes; contents need no initialisation; calls that share it
 *               must be ordered on one stream.  With BF16 qkv and at least
 *               kime_attn_workspace_bytes(3, ...) bytes, the qkv rows are
 *               first prepared into the workspace (a third launch: queries
 *               and keys rotated once each, queries scaled, all in FP16) and
 *               the attention kernel does no RoPE work: faster, with the same
 *               f16 operands and contract (its row sums add in another
 *               order, so the last bits of the output may differ).
 * BF16 runs on the tensor cores (tcgen05, FP32 accumulate) with f16 operands:
 * rotated keys, scaled rotated queries and values are rounded to f16, so they
 * must lie within its range (|x| <= 65504; beyond, they saturate and
 * KIME_DEV_RANGE is set).  FP32 qkv with
 * KIME_F32 / KIME_F32_F16OUT / KIME_F32_BF16OUT runs on FP32 FMA.  Launches:
 * the device scheduler, the row preparation when the workspace has room for
 * it, then the attention kernel.  KIME_F32_3XTF32 enqueues the scheduler and
 * one tensor-core kernel that reads the FP32 qkv rows itself (queries and keys
 * rotated, queries scaled, every operand split into TF32 high and low parts,
 * values transposed, all in shared memory and tensor memory). */
int kime_attn_varlen(const void* qkv, int dtype, const int32_t* cu_seqlens, int n_seqs, int total_tokens,
                     int max_seqlen, int heads, int kv_heads, int head_dim, int window, int causal, float scale,
                     const float* rope_cos, const float* rope_sin, int rope_len, void* out, void* workspace,
                     size_t workspace_bytes, int32_t* dev_status, void* stream);

/* kime_kv_append -- in-place KV-cache append of one new token per sequence
 * (ffai-argus KvAppend: rows written at pos, pos checked against cap before
 * any write).
 *
 *  qkv_new      device bf16 [n_seqs, W]: the new token's fused row per sequence
 *  pos          device int32 [n_seqs]: positions already used = the row written
 *  k_cache/v_cache  device bf16 [n_seqs, kv_heads, cap, 64]
 * Writes k_cache[s,g,pos[s]] = bf16(rope(k, pos[s])) (float32 rotation, one
 * rounding per operation, then round to nearest even) and v_cache[s,g,pos[s]] =
 * v.  Nothing else is written.  pos is not advanced (the caller does that).
 * pos[s] outside [0, min(cap, rope_len)) sets KIME_DEV_BAD_POS and skips s. */
int kime_kv_append(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                   int cap, const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache, void* v_cache,
                   int32_t* dev_status, void* stream);

/* kime_attn_decode -- single-token attention against the KV cache
 * (ffai-argus CausalSoftmax with q_len 1 and offset k_len-1: the new token
 * attends to the entire cache, rows 0..=pos[s], its own appended row included;
 * call kime_kv_append first).
 *
 *  qkv_new, pos, caches as for kime_kv_append (caches are read only)
 *  out          device bf16 [n_seqs, heads*64]
 *  workspace    device scratch of kime_attn_workspace_bytes(1, ...) bytes
 * Split-KV on the tensor cores: the keys 0..=pos[s] of each (sequence, kv
 * head) are cut into chunks of 128 keys and the chunks into work items of up
 * to 16; a one-CTA plan kernel lists the items (longest first) and zeroes the
 * per-(sequence, kv head) merge tickets, and a persistent decode kernel
 * (three CTAs per SM) streams each item's K/V tiles and reduces all q heads of
 * the kv group together; the last item of a (sequence, kv head) to finish
 * merges the partial results.  heads/kv_heads must be 1..8.  Two launches,
 * no memset. */
int kime_attn_decode(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                     int cap, float scale, const float* rope_cos, const float* rope_sin, int rope_len,
                     const void* k_cache, const void* v_cache, void* out, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream);

/* kime_decode_step -- kime_kv_append followed by kime_attn_decode in one
 * decode launch (after the plan kernel): the work item whose chunks hold row
 * pos[s] of a kv head writes the appended row (same rotation and rounding as
 * kime_kv_append) to the caches and uses it directly; no other item reads
 * that row.  Arguments as kime_attn_decode, with writable caches; workspace from
 * kime_attn_workspace_bytes(1, ...). */
int kime_decode_step(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                     int cap, float scale, const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache,
                     void* v_cache, void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream);

/* kime_kv_append_varlen -- multi-token in-place KV-cache append, the first
 * half of chunked prefill (ffai-argus 0.7.3 src/text.rs, TextTower::block: a
 * block of seq new tokens at index_pos is written into the preallocated cache,
 * KvAppend refusing pos + seq > cap before anything is written).
 *
 *  qkv          device bf16 [total_tokens, W], W = 64*(heads + 2*kv_heads):
 *               the new tokens, sequence s owning rows cu[s]..cu[s+1]-1
 *  cu_seqlens   device int32 [n_seqs+1], cu[0] = 0, cu[n_seqs] = total_tokens
 *  pos          device int32 [n_seqs]: cache rows already used; row i of
 *               sequence s is the token at position pos[s] + i
 *  k_cache/v_cache  device bf16 [n_seqs, kv_heads, cap, 64], 16-byte aligned
 * Writes k_cache[s,g,pos[s]+i] = bf16(rope(k, pos[s]+i)) (float32 rotation,
 * one rounding per operation, round to nearest even) and v_cache[s,g,pos[s]+i]
 * = v for every row; nothing else.  A sequence with pos[s] < 0 or
 * pos[s] + L > min(cap, rope_len) sets KIME_DEV_BAD_POS and none of its rows
 * is written; rows outside a valid cu set KIME_DEV_BAD_CU.  pos is not
 * advanced.  One launch. */
int kime_kv_append_varlen(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs,
                          int total_tokens, int heads, int kv_heads, int head_dim, int cap, const float* rope_cos,
                          const float* rope_sin, int rope_len, void* k_cache, void* v_cache, int32_t* dev_status,
                          void* stream);

/* kime_attn_chunk -- the attention half of chunked prefill: row i of sequence
 * s, at position P = pos[s] + i, attends cache rows 0..=P of its kv head
 * (ffai-argus CausalSoftmax: row i of a block at offset index_pos sees keys
 * 0..=i+offset).  The caches must already hold the chunk
 * (kime_kv_append_varlen on the same stream, or kime_chunk_step).  q is
 * rotated at P with the tables; cached keys are used as stored.
 *
 *  qkv, cu_seqlens, pos, caches  as for kime_kv_append_varlen (caches read only)
 *  max_seqlen   host upper bound on any chunk length (longer: KIME_DEV_SEQ_TOO_LONG)
 *  scale        softmax scale (> 0, finite)
 *  out          device bf16 [total_tokens, heads*64]
 *  workspace    device scratch of at least kime_attn_workspace_bytes(2, n_seqs,
 *               total_tokens, ...) bytes.  With kime_attn_workspace_bytes(5,
 *               n_seqs, total_tokens, heads, kv_heads, cap) bytes the chunk's
 *               queries are rotated and rounded to f16 once and cache rows
 *               0..pos[s]+L-1 widened to f16 once, in the workspace, and the
 *               attention runs over them (the faster path); with less, the
 *               attention kernel converts its own tiles.  Either gives
 *               results within the same bound.
 * BF16 inputs on the tensor cores, FP32 accumulation: the prefill kernels of
 * kime_attn_varlen with K/V tiles taken from the cache.  A sequence whose
 * positions leave [0, min(cap, rope_len)) sets KIME_DEV_BAD_POS and its rows
 * of out are not written; an operand beyond the f16 range sets
 * KIME_DEV_RANGE.  n_seqs*kv_heads*cap must stay below 2^31.  Launches:
 * scheduler and attention, with the op-5 workspace also the preparation
 * between them. */
int kime_attn_chunk(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                    int max_seqlen, int heads, int kv_heads, int head_dim, int cap, float scale,
                    const float* rope_cos, const float* rope_sin, int rope_len, const void* k_cache,
                    const void* v_cache, void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                    void* stream);

/* kime_chunk_step -- kime_kv_append_varlen then kime_attn_chunk on one stream
 * (three launches; with the op-5 workspace the preparation writes the
 * chunk's rows to the caches itself, the same bits, and no append kernel
 * runs).  Arguments as kime_attn_chunk, with writable caches. */
int kime_chunk_step(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                    int max_seqlen, int heads, int kv_heads, int head_dim, int cap, float scale,
                    const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache, void* v_cache,
                    void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Scratch bytes for op 0 (varlen, the minimum: uses n_seqs, total_tokens),
 * op 1 (decode: uses n_seqs, heads, kv_heads, cap), op 2 (chunked prefill:
 * uses n_seqs, total_tokens) or op 3 (varlen with room for the prepared qkv
 * rows, about total_tokens * 128 * (heads + 2 * kv_heads) bytes more: uses
 * n_seqs, total_tokens, heads, kv_heads) or op 4 (varlen with KIME_F32_3XTF32:
 * the size of op 0; heads and kv_heads are checked) or op 5 (chunked prefill
 * over prepared rows: op 2 plus the chunk's query rows, total_tokens * 128 *
 * heads bytes, and the widened cache rows, n_seqs * kv_heads * (cap rounded
 * up to a multiple of 128) * 256 bytes: uses all five sizes).  Returns 0 for
 * an unknown op or malformed sizes. */
size_t kime_attn_workspace_bytes(int op, int n_seqs, int total_tokens, int heads, int kv_heads, int cap);

/* kime_qkv_proj -- the QKV projection of a packed batch, the step before
 * attention: qkv = x W^T with one fused weight stored [out width, in width],
 * q rows, then k, then v (kime-cuda 0.0.3 src/plan.rs, Op::Gemm: weight shape
 * [out.width, a.width]; ffai-argus 0.7.3 src/text.rs, Block::q: the fused
 * [960, 576] weight of q, k and v).  No bias, no activation.
 *
 *  x            device bf16 [total_tokens, hidden], row-major, 16-byte aligned
 *  w            device bf16 [64*(heads + 2*kv_heads), hidden]
 *  hidden       a positive multiple of 64
 *  qkv          device bf16 [total_tokens, 64*(heads + 2*kv_heads)]: each value
 *               a sum of bf16 products accumulated in FP32 on the tensor cores,
 *               rounded to bf16 (nearest even)
 * One launch.  Returns KIME_EINVAL for bad shapes or pointers, KIME_ERANGE for
 * sizes beyond the library's index range. */
int kime_qkv_proj(const void* x, const void* w, int total_tokens, int hidden, int heads, int kv_heads,
                  int head_dim, void* qkv, int32_t* dev_status, void* stream);

/* kime_attn_varlen_proj -- kime_attn_varlen on BF16 qkv rows given by their
 * projection, qkv = x W^T (as kime_qkv_proj), with the projection fused into
 * the attention's producer: the projection's epilogue applies RoPE at each
 * token's position within its sequence, multiplies queries by
 * scale * log2(e) and rounds q, k and v once to f16 -- the prepared rows the
 * attention kernel loads -- from the FP32 accumulators, so no bf16 qkv is
 * written or read.  Arguments as kime_attn_varlen (dtype BF16 implied) plus
 * x, w and hidden as kime_qkv_proj; the workspace must hold
 * kime_attn_workspace_bytes(3, ...) bytes (KIME_ERANGE if less).  Launches:
 * the scheduler, the projection (beside it), the attention kernel.  An f16
 * operand beyond 65504 sets KIME_DEV_RANGE. */
int kime_attn_varlen_proj(const void* x, const void* w, const int32_t* cu_seqlens, int n_seqs, int total_tokens,
                          int hidden, int max_seqlen, int heads, int kv_heads, int head_dim, int window, int causal,
                          float scale, const float* rope_cos, const float* rope_sin, int rope_len, void* out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Host helper: float32 cos/sin tables [len, 32] for heads of 64 by kime-cuda's
 * fn rope_tables: inv_i = 1/(float)(theta^(float)(2i/64)) in float32, angle =
 * (float)p * inv_i in float32, cos and sin taken in double and narrowed.
 * cos_out / sin_out are HOST arrays of len*32 floats.  Returns KIME_EINVAL for
 * theta <= 0, len < 0 or null outputs. */
int kime_rope_tables(double theta, int len, float* cos_out, float* sin_out);

/* Test aid: run only the device scheduler of kime_attn_varlen and copy its
 * work list out.  tiles_out (device int32 [max_pairs, 8]) receives, per
 * (sequence, 128-row query tile) pair, {s, qt, kt_begin, kt_end, full_begin,
 * full_end, row0, L}: key tiles [kt_begin, kt_end) are visited and
 * [full_begin, full_end) need no per-key mask.  *n_pairs_out (device int32)
 * receives the count.  max_pairs must be >= total_tokens/128 + n_seqs + 1. */
int kime_attn_debug_tiles(const int32_t* cu_seqlens, int n_seqs, int total_tokens, int max_seqlen, int window,
                          int causal, void* workspace, size_t workspace_bytes, int32_t* tiles_out, int max_pairs,
                          int32_t* n_pairs_out, int32_t* dev_status, void* stream);

/* Test aid: kime_attn_debug_tiles for chunks at offsets pos (device int32
 * [n_seqs]) against a cache of cap rows: key tiles count cache rows from 0,
 * row i of sequence s sits at position pos[s] + i (causal). */
int kime_attn_debug_tiles_chunk(const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                                int max_seqlen, int cap, int rope_len, void* workspace, size_t workspace_bytes,
                                int32_t* tiles_out, int max_pairs, int32_t* n_pairs_out, int32_t* dev_status,
                                void* stream);

/* Bytes of the scratch array built into the library for kime_attn_varlen_noalloc. */
#define KIME_NOALLOC_SCRATCH_BYTES (1u << 20)

/* kime_attn_varlen_noalloc -- the same attention as kime_attn_varlen, for
 * callers that cannot allocate device memory when they call it (for instance a
 * host program whose own pool owns every device allocation, or a loop in which
 * an allocation, which may synchronise the device, is not allowed).  The source
 * pages have no counterpart of this entry point.
 *
 * Arguments are those of kime_attn_varlen without workspace / workspace_bytes:
 * the scheduler's scratch is a KIME_NOALLOC_SCRATCH_BYTES array inside the
 * library, held by every GPU that loads the library until the process exits.
 * Returns KIME_ERANGE, launching nothing, when the batch needs more scratch than
 * that (kime_attn_workspace_bytes(0, n_seqs, total_tokens, ...) is the need:
 * about 48 bytes per 128 tokens plus 64 per sequence, KIME_F32_3XTF32
 * included; a BF16 batch has its rows prepared only when they fit in the
 * array too).  The first
 * call on a device looks up the array's device address with that device
 * current; make it before any stream capture.  All calls share the array, so calls that
 * overlap on the GPU race; order them on one stream.  Allocates nothing. */
int kime_attn_varlen_noalloc(const void* qkv, int dtype, const int32_t* cu_seqlens, int n_seqs, int total_tokens,
                             int max_seqlen, int heads, int kv_heads, int head_dim, int window, int causal,
                             float scale, const float* rope_cos, const float* rope_sin, int rope_len, void* out,
                             int32_t* dev_status, void* stream);

/* The cudaError_t of the last failing CUDA call in this thread (0 if none). */
int kime_attn_last_cuda_error(void);

/* A static string naming a kime_status value. */
const char* kime_attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KIME_ATTN_H */
