// api.cu -- the C ABI of libkime_attn (declared in include/kime_attn.h):
// argument checks, workspace carving, TMA tensor-map encoding and launches.
// No allocation and no synchronisation happen here.
#include <math.h>
#include <string.h>

#include "../../include/kime_attn.h"
#include "kime_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KIME_OK;
  g_last_cuda_error = static_cast<int>(e);
  return KIME_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Mean sequence length under 2,048 tokens: the attention kernel over prepared
// rows then ends a unit every few key tiles, and the variant whose epilogue
// coalesces its stores is the faster one (ModernBERT-base, mean length 316:
// 0.0891 / 0.0932 ms for the local / global layer against 0.0932 / 0.0993;
// SmolLM2 prefill, 1,142: 0.0645 against 0.0706; ModernBERT-large global,
// 4,836: 1.0373 against 1.0271 ms, where the other one is kept).
int short_seqs(int n_seqs, int total_tokens) { return total_tokens < 2048LL * n_seqs ? 1 : 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over a bf16 row buffer [total, W] (the qkv rows, or a KV cache seen
// as [n_seqs*kv_heads*cap, 64]): boxes of 128 rows x 64 columns (one head of
// 128 tokens), 128-byte swizzle, rows past `total` read as zero.
int encode_qkv_map(CUtensorMap* map, const void* qkv, int total, int W) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KIME_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(total)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(W) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kime::kHead), static_cast<cuuint32_t>(kime::kBM)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int>(r);
    return KIME_ECUDA;
  }
  return KIME_OK;
}

// 2-D map over a bf16 row-major matrix [rows, cols]: boxes of 64 columns
// (128 bytes) x box_rows rows, 128-byte swizzle, elements past the ends read
// as zero.
int encode_bf16_map(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KIME_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int>(r);
    return KIME_ECUDA;
  }
  return KIME_OK;
}

// 2-D map over a RoPE table [rope_len, 32] f32: boxes of 128 rows (the
// positions of one key tile), 128-byte swizzle, rows past rope_len read as zero.
int encode_table_map(CUtensorMap* map, const float* table, int rope_len) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KIME_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kime::kHalf), static_cast<cuuint64_t>(rope_len > 0 ? rope_len : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kime::kHalf) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kime::kHalf), static_cast<cuuint32_t>(kime::kBN)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(table), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int>(r);
    return KIME_ECUDA;
  }
  return KIME_OK;
}

// 2-D map over an f32 matrix [rows, cols] (FP32 qkv rows for the 3xTF32
// path): boxes of box_rows rows x 32 columns (128 bytes), 128-byte swizzle,
// elements past either end read as zero.
int encode_f32_plane_map(CUtensorMap* map, const void* plane, long long cols, long long rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KIME_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(plane), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int>(r);
    return KIME_ECUDA;
  }
  return KIME_OK;
}

size_t varlen_ws_bytes(int n_seqs, int total) { return kime::varlen_workspace_bytes(n_seqs, total); }

// Workspace with room for the prepared qkv rows of a packed batch
// (launch_qkv_prep, [total, W] f16), placed after the scheduler's lists at a
// 1 KB boundary.
size_t prep_offset(int n_seqs, int total) { return (varlen_ws_bytes(n_seqs, total) + 1023) & ~static_cast<size_t>(1023); }
size_t prep_ws_bytes(int n_seqs, int total, int heads, int kv_heads) {
  return prep_offset(n_seqs, total) + static_cast<size_t>(total) * kime::kHead * (heads + 2 * kv_heads) * 2;
}

// Workspace of the chunked prefill over prepared rows (launch_chunk_prep):
// the scheduler's lists, then at 1 KB boundaries the chunk's prepared query
// rows [total, heads*64] f16 and the widened cache rows [n_seqs * kv_heads *
// cap_pad, 128] f16, cap_pad = cap rounded up to whole 128-key tiles (so no
// key tile of one kv head reaches into the next).
int cap_pad_for(int cap) { return (cap + kime::kBN - 1) / kime::kBN * kime::kBN; }
size_t chunk_kv16_offset(int n_seqs, int total, int heads) {
  return (prep_offset(n_seqs, total) + static_cast<size_t>(total) * kime::kHead * heads * 2 + 1023) &
         ~static_cast<size_t>(1023);
}
size_t chunk_prep_ws_bytes(int n_seqs, int total, int heads, int kv_heads, int cap) {
  return chunk_kv16_offset(n_seqs, total, heads) +
         static_cast<size_t>(n_seqs) * kv_heads * cap_pad_for(cap) * 2 * kime::kHead * 2;
}

bool heads_ok(int heads, int kv_heads, int head_dim) {
  return head_dim == kime::kHead && heads > 0 && kv_heads > 0 && heads % kv_heads == 0;
}

}  // namespace

void kime::set_last_cuda_error(int e) { g_last_cuda_error = e; }

extern "C" {

size_t kime_attn_workspace_bytes(int op, int n_seqs, int total_tokens, int heads, int kv_heads, int cap) {
  if (n_seqs < 0) return 0;
  if (op == 0) {
    if (total_tokens < 0) return 0;
    return varlen_ws_bytes(n_seqs, total_tokens);
  }
  if (op == 1) {
    if (!heads_ok(heads, kv_heads, kime::kHead) || cap <= 0) return 0;
    return kime::decode_workspace_bytes(n_seqs, heads, kv_heads, cap);
  }
  if (op == 2) {
    if (total_tokens < 0) return 0;
    return varlen_ws_bytes(n_seqs, total_tokens);
  }
  if (op == 3) {
    if (total_tokens < 0 || !heads_ok(heads, kv_heads, kime::kHead)) return 0;
    return prep_ws_bytes(n_seqs, total_tokens, heads, kv_heads);
  }
  if (op == 4) {  // the 3xTF32 path needs no more scratch than op 0
    if (total_tokens < 0 || !heads_ok(heads, kv_heads, kime::kHead)) return 0;
    return varlen_ws_bytes(n_seqs, total_tokens);
  }
  if (op == 5) {  // chunked prefill over prepared rows
    if (total_tokens < 0 || !heads_ok(heads, kv_heads, kime::kHead) || cap <= 0 || cap > (1 << 30)) return 0;
    return chunk_prep_ws_bytes(n_seqs, total_tokens, heads, kv_heads, cap);
  }
  return 0;
}

int kime_attn_varlen(const void* qkv, int dtype, const int32_t* cu_seqlens, int n_seqs, int total_tokens,
                     int max_seqlen, int heads, int kv_heads, int head_dim, int window, int causal, float scale,
                     const float* rope_cos, const float* rope_sin, int rope_len, void* out, void* workspace,
                     size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (dtype != KIME_F32 && dtype != KIME_BF16 && dtype != KIME_F32_F16OUT && dtype != KIME_F32_BF16OUT &&
      dtype != KIME_F32_3XTF32)
    return KIME_EINVAL;
  if (!heads_ok(heads, kv_heads, head_dim)) return KIME_EINVAL;
  if (n_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || rope_len < 0 || window < -1) return KIME_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return KIME_EINVAL;
  if (causal != 0 && causal != 1) return KIME_EINVAL;
  if (n_seqs == 0 || total_tokens == 0) return KIME_OK;
  if (!qkv || !cu_seqlens || !rope_cos || !rope_sin || !out || !workspace) return KIME_EINVAL;
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(rope_cos) || !aligned16(rope_sin) || !aligned16(workspace))
    return KIME_EINVAL;
  if (max_seqlen > rope_len) return KIME_ERANGE;
  if (workspace_bytes < varlen_ws_bytes(n_seqs, total_tokens)) return KIME_ERANGE;
  const long long W = 64LL * (heads + 2LL * kv_heads);
  if (W > (1LL << 30) || static_cast<long long>(total_tokens) * W > (1LL << 46)) return KIME_ERANGE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int max_pairs = kime::max_pairs_for(n_seqs, total_tokens);
  int rc;
  if (dtype == KIME_F32_3XTF32) {
    // FP32 on the tensor cores: the scheduler, then the attention kernel on the raw qkv rows
    CUtensorMap qmap;
    if ((rc = encode_f32_plane_map(&qmap, qkv, W, total_tokens, 64))) return rc;
    if ((rc = cuda_status(kime::launch_schedule(cu_seqlens, nullptr, n_seqs, total_tokens, max_seqlen, causal,
                                                window, 0, 0, workspace, max_pairs, dev_status, st))))
      return rc;
    return cuda_status(kime::launch_prefill_3xtf32(&qmap, heads, kv_heads, window, causal, scale, rope_cos, rope_sin,
                                                   static_cast<float*>(out), workspace, dev_status, st));
  }
  rc = cuda_status(kime::launch_schedule(cu_seqlens, nullptr, n_seqs, total_tokens, max_seqlen, causal, window,
                                         0, 0, workspace, max_pairs, dev_status, st));
  if (rc) return rc;
  if (dtype != KIME_BF16) {
    const int out_kind = dtype == KIME_F32 ? 0 : (dtype == KIME_F32_F16OUT ? 1 : 2);
    return cuda_status(kime::launch_varlen_f32(static_cast<const float*>(qkv), cu_seqlens, n_seqs, total_tokens,
                                               heads, kv_heads, window, causal, scale, rope_cos, rope_sin, out,
                                               out_kind, workspace, max_pairs, dev_status, st));
  }
  CUtensorMap map, cmap, smap, pmap;
  if ((rc = encode_qkv_map(&map, qkv, total_tokens, static_cast<int>(W)))) return rc;
  // With room in the workspace, the rows are prepared once (RoPE and f16) and
  // the attention kernel does no RoPE work: the faster way for every layer
  // measured (ModernBERT-large local layer, window 64: 0.169 ms against 0.184
  // for the kernel that rotates its own tiles; the global layers and short
  // sequences by more).
  const bool prep = workspace_bytes >= prep_ws_bytes(n_seqs, total_tokens, heads, kv_heads);
  if (prep) {
    void* rows = static_cast<char*>(workspace) + prep_offset(n_seqs, total_tokens);
    if ((rc = encode_qkv_map(&pmap, rows, total_tokens, static_cast<int>(W)))) return rc;
    if ((rc = cuda_status(kime::launch_qkv_prep(qkv, cu_seqlens, n_seqs, total_tokens, heads, kv_heads, scale,
                                                rope_cos, rope_sin, rope_len, rows, dev_status, st))))
      return rc;
  } else {
    if ((rc = encode_table_map(&cmap, rope_cos, rope_len))) return rc;
    if ((rc = encode_table_map(&smap, rope_sin, rope_len))) return rc;
  }
  if (prep)
    return cuda_status(kime::launch_prefill_rows(&pmap, heads, kv_heads, window, causal, out, workspace, max_pairs,
                                                 short_seqs(n_seqs, total_tokens), dev_status, st));
  return cuda_status(kime::launch_prefill_tc(&map, nullptr, nullptr, &cmap, &smap, heads, kv_heads, 0, window,
                                             causal, scale, rope_cos, rope_sin, out, workspace, max_pairs,
                                             short_seqs(n_seqs, total_tokens), dev_status, st));
}

int kime_qkv_proj(const void* x, const void* w, int total_tokens, int hidden, int heads, int kv_heads,
                  int head_dim, void* qkv, int32_t* dev_status, void* stream) {
  if (!heads_ok(heads, kv_heads, head_dim) || total_tokens < 0 || hidden <= 0 || hidden % 64 != 0)
    return KIME_EINVAL;
  if (total_tokens == 0) return KIME_OK;
  if (!x || !w || !qkv || !aligned16(x) || !aligned16(w) || !aligned16(qkv)) return KIME_EINVAL;
  const long long W = 64LL * (heads + 2LL * kv_heads);
  if (W > (1LL << 30) || static_cast<long long>(total_tokens) * (W > hidden ? W : hidden) > (1LL << 46))
    return KIME_ERANGE;
  CUtensorMap xm, wm;
  int rc;
  if ((rc = encode_bf16_map(&xm, x, total_tokens, hidden, kime::kBM))) return rc;
  if ((rc = encode_bf16_map(&wm, w, W, hidden, 256))) return rc;
  return cuda_status(kime::launch_qkv_proj(&xm, &wm, total_tokens, hidden, heads, kv_heads, nullptr, 0, 1.f,
                                           nullptr, nullptr, 0, qkv, 1, dev_status,
                                           static_cast<cudaStream_t>(stream)));
}

int kime_attn_varlen_proj(const void* x, const void* w, const int32_t* cu_seqlens, int n_seqs, int total_tokens,
                          int hidden, int max_seqlen, int heads, int kv_heads, int head_dim, int window, int causal,
                          float scale, const float* rope_cos, const float* rope_sin, int rope_len, void* out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!heads_ok(heads, kv_heads, head_dim) || hidden <= 0 || hidden % 64 != 0) return KIME_EINVAL;
  if (n_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || rope_len < 0 || window < -1) return KIME_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return KIME_EINVAL;
  if (causal != 0 && causal != 1) return KIME_EINVAL;
  if (n_seqs == 0 || total_tokens == 0) return KIME_OK;
  if (!x || !w || !cu_seqlens || !rope_cos || !rope_sin || !out || !workspace) return KIME_EINVAL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned16(rope_cos) || !aligned16(rope_sin) ||
      !aligned16(workspace))
    return KIME_EINVAL;
  if (max_seqlen > rope_len) return KIME_ERANGE;
  const long long W = 64LL * (heads + 2LL * kv_heads);
  if (W > (1LL << 30) || static_cast<long long>(total_tokens) * (W > hidden ? W : hidden) > (1LL << 46))
    return KIME_ERANGE;
  if (workspace_bytes < prep_ws_bytes(n_seqs, total_tokens, heads, kv_heads)) return KIME_ERANGE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int max_pairs = kime::max_pairs_for(n_seqs, total_tokens);
  void* rows = static_cast<char*>(workspace) + prep_offset(n_seqs, total_tokens);
  CUtensorMap xm, wm, pmap;
  int rc;
  if ((rc = encode_bf16_map(&xm, x, total_tokens, hidden, kime::kBM))) return rc;
  if ((rc = encode_bf16_map(&wm, w, W, hidden, 256))) return rc;
  if ((rc = encode_qkv_map(&pmap, rows, total_tokens, static_cast<int>(W)))) return rc;
  // scheduler, then the projection writing the prepared rows beside it, then
  // the attention kernel over them
  if ((rc = cuda_status(kime::launch_schedule(cu_seqlens, nullptr, n_seqs, total_tokens, max_seqlen, causal,
                                              window, 0, 0, workspace, max_pairs, dev_status, st))))
    return rc;
  if ((rc = cuda_status(kime::launch_qkv_proj(&xm, &wm, total_tokens, hidden, heads, kv_heads, cu_seqlens, n_seqs,
                                              scale, rope_cos, rope_sin, rope_len, rows, 0, dev_status, st))))
    return rc;
  return cuda_status(kime::launch_prefill_rows(&pmap, heads, kv_heads, window, causal, out, workspace, max_pairs,
                                               short_seqs(n_seqs, total_tokens), dev_status, st));
}

int kime_kv_append(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                   int cap, const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache, void* v_cache,
                   int32_t* dev_status, void* stream) {
  if (!heads_ok(heads, kv_heads, head_dim) || n_seqs < 0 || cap <= 0 || rope_len < 0) return KIME_EINVAL;
  if (n_seqs == 0) return KIME_OK;
  if (!qkv_new || !pos || !rope_cos || !rope_sin || !k_cache || !v_cache) return KIME_EINVAL;
  if (n_seqs > (1 << 30)) return KIME_ERANGE;
  return cuda_status(kime::launch_kv_append(qkv_new, pos, n_seqs, heads, kv_heads, cap, rope_cos, rope_sin,
                                            rope_len, k_cache, v_cache, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Host checks shared by the chunked-prefill entry points (append: out and
// workspace unused).
int chunk_args_ok(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total, int heads,
                  int kv_heads, int head_dim, int cap, const float* rope_cos, const float* rope_sin, int rope_len,
                  const void* k_cache, const void* v_cache) {
  if (!heads_ok(heads, kv_heads, head_dim) || n_seqs < 0 || total < 0 || cap <= 0 || rope_len < 0)
    return KIME_EINVAL;
  if (n_seqs == 0 || total == 0) return KIME_OK;
  if (!qkv || !cu || !pos || !rope_cos || !rope_sin || !k_cache || !v_cache) return KIME_EINVAL;
  if (!aligned16(qkv) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(rope_cos) || !aligned16(rope_sin))
    return KIME_EINVAL;
  const long long W = 64LL * (heads + 2LL * kv_heads);
  if (W > (1LL << 30) || static_cast<long long>(total) * W > (1LL << 46)) return KIME_ERANGE;
  if (static_cast<long long>(n_seqs) * kv_heads * cap >= (1LL << 31)) return KIME_ERANGE;
  return KIME_OK;
}

// With room in the workspace the chunk's queries are prepared and the visible
// cache rows widened to f16 once, and the attention kernel over prepared rows
// takes them (SmolLM2 chunked prefill step: 0.251 ms against 0.320 for the
// kernel that converts its own tiles); else that kernel.
bool chunk_prep_fits(int n_seqs, int total, int heads, int kv_heads, int cap, size_t workspace_bytes) {
  return workspace_bytes >= chunk_prep_ws_bytes(n_seqs, total, heads, kv_heads, cap) &&
         static_cast<long long>(n_seqs) * kv_heads * cap_pad_for(cap) < (1LL << 31);
}

// append (the chunk step over prepared rows only): the preparation also writes
// the chunk's rows to the caches.
int chunk_attend(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total, int max_seqlen,
                 int heads, int kv_heads, int cap, float scale, const float* rope_cos, const float* rope_sin,
                 int rope_len, const void* k_cache, const void* v_cache, void* out, void* workspace, bool prep,
                 bool append, int32_t* dev_status, cudaStream_t st) {
  const int max_pairs = kime::max_pairs_for(n_seqs, total);
  int rc = cuda_status(kime::launch_schedule(cu, pos, n_seqs, total, max_seqlen, 1, -1, cap, rope_len, workspace,
                                             max_pairs, dev_status, st));
  if (rc) return rc;
  const int cap_pad = cap_pad_for(cap);
  if (prep) {
    void* q16 = static_cast<char*>(workspace) + prep_offset(n_seqs, total);
    void* kv16 = static_cast<char*>(workspace) + chunk_kv16_offset(n_seqs, total, heads);
    CUtensorMap qmap, kvmap;
    if ((rc = encode_qkv_map(&qmap, q16, total, 64 * heads))) return rc;
    if ((rc = encode_qkv_map(&kvmap, kv16, n_seqs * kv_heads * cap_pad, 2 * kime::kHead))) return rc;
    if ((rc = cuda_status(kime::launch_chunk_prep(qkv, cu, pos, n_seqs, total, heads, kv_heads, cap, cap_pad, scale,
                                                  rope_cos, rope_sin, rope_len, const_cast<void*>(k_cache),
                                                  const_cast<void*>(v_cache), append ? 1 : 0, q16, kv16,
                                                  dev_status, st))))
      return rc;
    return cuda_status(kime::launch_prefill_rows_chunk(&qmap, &kvmap, heads, kv_heads, cap_pad, out, workspace,
                                                       max_pairs, dev_status, st));
  }
  const int W = 64 * (heads + 2 * kv_heads), rows = n_seqs * kv_heads * cap;
  CUtensorMap qmap, kmap, vmap;
  if ((rc = encode_qkv_map(&qmap, qkv, total, W))) return rc;
  if ((rc = encode_qkv_map(&kmap, k_cache, rows, kime::kHead))) return rc;
  if ((rc = encode_qkv_map(&vmap, v_cache, rows, kime::kHead))) return rc;
  return cuda_status(kime::launch_prefill_tc(&qmap, &kmap, &vmap, nullptr, nullptr, heads, kv_heads, cap, -1, 1, scale,
                                             rope_cos, rope_sin, out, workspace, max_pairs, 0, dev_status, st));
}

int chunk_common(const void* qkv, const int32_t* cu, const int32_t* pos, int n_seqs, int total, int max_seqlen,
                 int heads, int kv_heads, int head_dim, int cap, float scale, const float* rope_cos,
                 const float* rope_sin, int rope_len, const void* k_cache, const void* v_cache, void* out,
                 void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream, bool append) {
  int rc = chunk_args_ok(qkv, cu, pos, n_seqs, total, heads, kv_heads, head_dim, cap, rope_cos, rope_sin, rope_len,
                         k_cache, v_cache);
  if (rc) return rc;
  if (!(scale > 0.f) || !isfinite(scale) || max_seqlen < 0) return KIME_EINVAL;
  if (n_seqs == 0 || total == 0) return KIME_OK;
  if (!out || !workspace || !aligned16(out) || !aligned16(workspace)) return KIME_EINVAL;
  if (workspace_bytes < varlen_ws_bytes(n_seqs, total)) return KIME_ERANGE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool prep = chunk_prep_fits(n_seqs, total, heads, kv_heads, cap, workspace_bytes);
  if (append && !prep) {
    rc = cuda_status(kime::launch_kv_append_varlen(qkv, cu, pos, n_seqs, total, heads, kv_heads, cap, rope_cos,
                                                   rope_sin, rope_len, const_cast<void*>(k_cache),
                                                   const_cast<void*>(v_cache), dev_status, st));
    if (rc) return rc;
  }
  return chunk_attend(qkv, cu, pos, n_seqs, total, max_seqlen, heads, kv_heads, cap, scale, rope_cos, rope_sin,
                      rope_len, k_cache, v_cache, out, workspace, prep, append && prep, dev_status, st);
}

int decode_common(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim, int cap,
                  float scale, const float* rope_cos, const float* rope_sin, int rope_len, const void* k_cache,
                  const void* v_cache, void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                  void* stream, bool append) {
  if (!heads_ok(heads, kv_heads, head_dim) || n_seqs < 0 || cap <= 0 || rope_len < 0) return KIME_EINVAL;
  if (heads / kv_heads > kime::kMaxGroup) return KIME_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return KIME_EINVAL;
  if (n_seqs == 0) return KIME_OK;
  if (!qkv_new || !pos || !rope_cos || !rope_sin || !k_cache || !v_cache || !out || !workspace) return KIME_EINVAL;
  if (!aligned16(qkv_new) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace) || !aligned16(out) ||
      !aligned16(rope_cos) || !aligned16(rope_sin))
    return KIME_EINVAL;
  if (n_seqs > 65535) return KIME_ERANGE;
  if (static_cast<long long>(kime::dec_items_for(cap)) * n_seqs * kv_heads >= (1LL << 30)) return KIME_ERANGE;
  if (workspace_bytes < kime::decode_workspace_bytes(n_seqs, heads, kv_heads, cap)) return KIME_ERANGE;
  if (static_cast<long long>(n_seqs) * kv_heads * cap >= (1LL << 31)) return KIME_ERANGE;
  CUtensorMap kmap, vmap;
  const int rows = n_seqs * kv_heads * cap;
  int rc = encode_qkv_map(&kmap, k_cache, rows, kime::kHead);
  if (rc) return rc;
  if ((rc = encode_qkv_map(&vmap, v_cache, rows, kime::kHead))) return rc;
  return cuda_status(kime::launch_decode(&kmap, &vmap, qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, rope_cos, rope_sin,
                                         rope_len, k_cache, v_cache, out, workspace, dev_status,
                                         static_cast<cudaStream_t>(stream), append));
}

}  // namespace

extern "C" {

int kime_attn_decode(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                     int cap, float scale, const float* rope_cos, const float* rope_sin, int rope_len,
                     const void* k_cache, const void* v_cache, void* out, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream) {
  return decode_common(qkv_new, pos, n_seqs, heads, kv_heads, head_dim, cap, scale, rope_cos, rope_sin, rope_len,
                       k_cache, v_cache, out, workspace, workspace_bytes, dev_status, stream, false);
}

int kime_decode_step(const void* qkv_new, const int32_t* pos, int n_seqs, int heads, int kv_heads, int head_dim,
                     int cap, float scale, const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache,
                     void* v_cache, void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream) {
  return decode_common(qkv_new, pos, n_seqs, heads, kv_heads, head_dim, cap, scale, rope_cos, rope_sin, rope_len,
                       k_cache, v_cache, out, workspace, workspace_bytes, dev_status, stream, true);
}

int kime_kv_append_varlen(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs,
                          int total_tokens, int heads, int kv_heads, int head_dim, int cap, const float* rope_cos,
                          const float* rope_sin, int rope_len, void* k_cache, void* v_cache, int32_t* dev_status,
                          void* stream) {
  int rc = chunk_args_ok(qkv, cu_seqlens, pos, n_seqs, total_tokens, heads, kv_heads, head_dim, cap, rope_cos,
                         rope_sin, rope_len, k_cache, v_cache);
  if (rc || n_seqs == 0 || total_tokens == 0) return rc;
  return cuda_status(kime::launch_kv_append_varlen(qkv, cu_seqlens, pos, n_seqs, total_tokens, heads, kv_heads, cap,
                                                   rope_cos, rope_sin, rope_len, k_cache, v_cache, dev_status,
                                                   static_cast<cudaStream_t>(stream)));
}

int kime_attn_chunk(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                    int max_seqlen, int heads, int kv_heads, int head_dim, int cap, float scale,
                    const float* rope_cos, const float* rope_sin, int rope_len, const void* k_cache,
                    const void* v_cache, void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                    void* stream) {
  return chunk_common(qkv, cu_seqlens, pos, n_seqs, total_tokens, max_seqlen, heads, kv_heads, head_dim, cap, scale,
                      rope_cos, rope_sin, rope_len, k_cache, v_cache, out, workspace, workspace_bytes, dev_status,
                      stream, false);
}

int kime_chunk_step(const void* qkv, const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                    int max_seqlen, int heads, int kv_heads, int head_dim, int cap, float scale,
                    const float* rope_cos, const float* rope_sin, int rope_len, void* k_cache, void* v_cache,
                    void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return chunk_common(qkv, cu_seqlens, pos, n_seqs, total_tokens, max_seqlen, heads, kv_heads, head_dim, cap, scale,
                      rope_cos, rope_sin, rope_len, k_cache, v_cache, out, workspace, workspace_bytes, dev_status,
                      stream, true);
}

int kime_rope_tables(double theta, int len, float* cos_out, float* sin_out) {
  if (!(theta > 0.0) || len < 0 || (len > 0 && (!cos_out || !sin_out))) return KIME_EINVAL;
  float inv[kime::kHalf];
  for (int i = 0; i < kime::kHalf; ++i) {
    const float expo = static_cast<float>(2 * i) / static_cast<float>(kime::kHead);
    inv[i] = 1.0f / static_cast<float>(pow(theta, static_cast<double>(expo)));
  }
  for (int p = 0; p < len; ++p) {
    for (int i = 0; i < kime::kHalf; ++i) {
      const double a = static_cast<double>(static_cast<float>(p) * inv[i]);
      cos_out[static_cast<size_t>(p) * kime::kHalf + i] = static_cast<float>(cos(a));
      sin_out[static_cast<size_t>(p) * kime::kHalf + i] = static_cast<float>(sin(a));
    }
  }
  return KIME_OK;
}

}  // extern "C"

namespace {

int debug_tiles_common(const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens, int max_seqlen,
                       int window, int causal, int cap, int rope_len, void* workspace, size_t workspace_bytes,
                       int32_t* tiles_out, int max_pairs, int32_t* n_pairs_out, int32_t* dev_status, void* stream) {
  if (n_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || window < -1) return KIME_EINVAL;
  if (!cu_seqlens || !workspace || !tiles_out || !n_pairs_out) return KIME_EINVAL;
  const int need = kime::max_pairs_for(n_seqs, total_tokens);
  if (max_pairs < need || workspace_bytes < varlen_ws_bytes(n_seqs, total_tokens)) return KIME_ERANGE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = cuda_status(kime::launch_schedule(cu_seqlens, pos, n_seqs, total_tokens, max_seqlen, causal ? 1 : 0,
                                             window, cap, rope_len, workspace, need, dev_status, st));
  if (rc) return rc;
  const char* ws = static_cast<const char*>(workspace);
  rc = cuda_status(cudaMemcpyAsync(n_pairs_out, ws + offsetof(kime::WsHeader, n_pairs), 4,
                                   cudaMemcpyDeviceToDevice, st));
  if (rc) return rc;
  return cuda_status(cudaMemcpyAsync(tiles_out, ws + sizeof(kime::WsHeader), static_cast<size_t>(need) * 32,
                                     cudaMemcpyDeviceToDevice, st));
}

}  // namespace

extern "C" {

int kime_attn_debug_tiles(const int32_t* cu_seqlens, int n_seqs, int total_tokens, int max_seqlen, int window,
                          int causal, void* workspace, size_t workspace_bytes, int32_t* tiles_out, int max_pairs,
                          int32_t* n_pairs_out, int32_t* dev_status, void* stream) {
  return debug_tiles_common(cu_seqlens, nullptr, n_seqs, total_tokens, max_seqlen, window, causal, 0, 0, workspace,
                            workspace_bytes, tiles_out, max_pairs, n_pairs_out, dev_status, stream);
}

int kime_attn_debug_tiles_chunk(const int32_t* cu_seqlens, const int32_t* pos, int n_seqs, int total_tokens,
                                int max_seqlen, int cap, int rope_len, void* workspace, size_t workspace_bytes,
                                int32_t* tiles_out, int max_pairs, int32_t* n_pairs_out, int32_t* dev_status,
                                void* stream) {
  if (!pos || cap <= 0 || rope_len < 0) return KIME_EINVAL;
  return debug_tiles_common(cu_seqlens, pos, n_seqs, total_tokens, max_seqlen, -1, 1, cap, rope_len, workspace,
                            workspace_bytes, tiles_out, max_pairs, n_pairs_out, dev_status, stream);
}

int kime_attn_last_cuda_error(void) { return g_last_cuda_error; }

const char* kime_attn_status_string(int status) {
  switch (status) {
    case KIME_OK: return "ok";
    case KIME_EINVAL: return "invalid argument";
    case KIME_ERANGE: return "size out of range";
    case KIME_ECUDA: return "CUDA error";
    case KIME_ETIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
