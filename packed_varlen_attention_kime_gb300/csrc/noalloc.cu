// noalloc.cu -- kime_attn_varlen_noalloc: the packed-varlen attention entry
// point for callers that cannot allocate device memory when they call it.
//
// kime_attn_varlen needs a small caller-provided scratch buffer (the device
// scheduler's work list).  Some callers have no way to provide one: a host
// program that hands every byte of device memory to its own pool at start-up
// and lets plug-ins allocate nothing afterwards, or a latency-critical loop in
// which an allocation -- which may synchronise the device -- is not allowed.
// This entry point takes its scratch from a fixed array that lives in the
// library itself, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the library
// holds it (kNoAllocScratchBytes) until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress while that device is current
// and keeps it; make that first call on a device before any stream capture.
// Every call shares the one array: calls that overlap on the GPU (other
// streams, other host threads) race on it and must be ordered by the caller.
// The scheduler rewrites every field it reads (the work counters start at zero
// on each call), so nothing left by an earlier call leaks into the next.
#include <atomic>

#include "../../include/kime_attn.h"
#include "kime_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = KIME_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" int kime_attn_varlen_noalloc(const void* qkv, int dtype, const int32_t* cu_seqlens, int n_seqs,
                                        int total_tokens, int max_seqlen, int heads, int kv_heads, int head_dim,
                                        int window, int causal, float scale, const float* rope_cos,
                                        const float* rope_sin, int rope_len, void* out, int32_t* dev_status,
                                        void* stream) {
  if (n_seqs < 0 || total_tokens < 0) return KIME_EINVAL;
  const size_t need = kime_attn_workspace_bytes(0, n_seqs, total_tokens, heads, kv_heads, 1);
  if (need > kNoAllocScratchBytes) return KIME_ERANGE;  // batch too large for the built-in scratch
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    kime::set_last_cuda_error(static_cast<int>(e));
    return KIME_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return KIME_ERANGE;  // more devices than the address table holds
  void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || !scratch) {
      kime::set_last_cuda_error(static_cast<int>(e));
      return KIME_ECUDA;
    }
    g_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  return kime_attn_varlen(qkv, dtype, cu_seqlens, n_seqs, total_tokens, max_seqlen, heads, kv_heads, head_dim,
                          window, causal, scale, rope_cos, rope_sin, rope_len, out, scratch, kNoAllocScratchBytes,
                          dev_status, stream);
}
