// pa_decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// pa_decode needs a few MB of scratch (per-CTA partial results and a
// per-sequence prefix) and asks the caller for it.  Some callers have no way
// to provide that: code embedded in a host program that owns no device
// allocator, code that must not call cudaMalloc on its path (the call can
// synchronise the whole device and stall other streams), or code running
// under a framework that has already reserved all device memory for its own
// pool.  This entry point serves them with scratch that lives in a fixed-size
// static device array of this library instead.
//
// The array belongs to the library's device image: every GPU that loads the
// library holds its kStaticScratchBytes until the process exits.  Every call
// on a device uses the same array, so two calls whose kernels overlap on the
// GPU (different streams, no ordering between them) corrupt each other's
// scratch; calls on one stream, or otherwise ordered, are safe.  The array
// starts zeroed (static device storage), which is what pa_decode's workspace
// contract asks for, and each call leaves its counters at zero again.
#include <mutex>

#include "pa_common.cuh"

namespace pagedkv {

// Upper bound of the scratch this entry point can use (bytes).
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

// The scratch itself.  In host code this name stands for the array but is not
// its device address: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device, looked up once
// per device (the lookup loads this library's device image there if needed).
static pa_status static_scratch_address(void **out) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no sticky error behind for the caller
      return PA_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return PA_OK;
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *block_tables, int max_blocks_per_seq,
                                       const int32_t *context_lens, int num_seqs, int num_heads,
                                       int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                       float scale, pa_dtype dtype, int *debug_err, void *stream) {
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return PA_ERR_WORKSPACE;  // more scratch than the static array holds
  void *scratch = nullptr;
  const pa_status st = static_scratch_address(&scratch);
  if (st != PA_OK) return st;
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, scratch, kStaticScratchBytes,
                   debug_err, stream);
}
