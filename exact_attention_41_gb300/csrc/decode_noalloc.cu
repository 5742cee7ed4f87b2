// attn_fwd_kvcache_noalloc: paged decode whose split scratch lives in a
// fixed array inside this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// code that runs while a CUDA graph is being captured (cudaMalloc is not a
// capturable operation), plugins of inference servers whose device memory is
// owned by a pool they cannot grow, and C hosts that have no CUDA allocator
// of their own.  They pass only inputs and outputs; the partial results of
// the key-range splits go to g_noalloc_scratch below.
#include <mutex>

#include "kernels.h"

namespace attn {
namespace {

// Upper bound of the scratch: split partial outputs (fp32) plus their LSEs.
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol is only a host-side stand-in, so the address is looked up once
// per device, with that device current.
void *scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace attn

extern "C" {

attn_status attn_fwd_kvcache_noalloc(const void *q, void *k_cache, void *v_cache,
                                     const void *k_new, const void *v_new,
                                     const int32_t *cache_seqlens, const int32_t *block_table,
                                     int num_pages, int page_size, int max_pages_per_seq,
                                     void *out, float *lse, int dtype, int b, int sq, int s_new,
                                     int hq, int hkv, int d, float scale, int causal, int win_l,
                                     int win_r, float softcap, int num_splits,
                                     attn_stream_t stream) {
  if (page_size <= 0 || max_pages_per_seq <= 0 || num_splits < 0)
    return ATTN_ERR_INVALID;
  const int64_t cap = (int64_t)max_pages_per_seq * page_size;
  if (cap > INT32_MAX / 2) return ATTN_ERR_UNSUPPORTED;
  const size_t need =
      attn_kvcache_workspace_size(b, sq, hq, hkv, d, (int)cap, num_splits);
  if (need > attn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  void *scratch = attn::scratch_address();
  if (!scratch) return ATTN_ERR_CUDA;
  return attn_fwd_kvcache(q, k_cache, v_cache, k_new, v_new, cache_seqlens, block_table,
                          num_pages, page_size, max_pages_per_seq, out, lse, dtype, b, sq, s_new,
                          hq, hkv, d, scale, causal, win_l, win_r, softcap, num_splits, scratch,
                          attn::kNoAllocScratchBytes, stream);
}

}  // extern "C"
