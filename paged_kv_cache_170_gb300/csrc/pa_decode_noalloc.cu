// pa_decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// pa_decode needs a few MB of scratch (per-CTA partial results and per-pair
// arrival counters) and asks the caller for it.  Some callers have no way to
// provide that: code embedded in a host program that owns no device
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
// scratch; calls on one stream, or otherwise ordered, are safe.  Each call
// first clears the array's counter region on its stream (cudaMemsetAsync,
// which allocates nothing), so a call never depends on what an earlier call
// left there, not even one that reported PA_DEVERR_TIMEOUT.
#include "pa_common.cuh"

namespace pagedkv {

// Defined with the decode (pa_decode.cu): byte offset and size of the
// per-pair counters in a decode workspace on the current device, and the
// host-side checks pa_decode makes before it launches anything.
bool decode_counter_region(int num_seqs, int num_heads, int head_dim, size_t *offset, size_t *bytes);
struct DecodeShape;
pa_status check_decode_call(const void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, float scale, pa_dtype dtype, const void *workspace,
                            DecodeShape *shape);

// Upper bound of the scratch this entry point can use (bytes).
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

// The scratch itself.  In host code this name stands for the array but is not
// its device address: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device.  Looked up on
// every call (cheap once the library's device code is loaded there), so an
// address never outlives the context it was taken in (cudaDeviceReset, a
// different current context).  The first lookup on a device may load the
// library's device code there.
static pa_status static_scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // leave no sticky error behind for the caller
    return PA_ERR_CUDA;
  }
  *out = p;
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
  size_t ctr_offset = 0, ctr_bytes = 0;
  if (!decode_counter_region(num_seqs, num_heads, head_dim, &ctr_offset, &ctr_bytes)) return PA_ERR_INVALID_ARG;
  if (ctr_offset + ctr_bytes > kStaticScratchBytes) return PA_ERR_WORKSPACE;
  void *scratch = nullptr;
  pa_status st = static_scratch_address(&scratch);
  if (st != PA_OK) return st;
  // arguments pa_decode would refuse are refused before anything is enqueued
  st = check_decode_call(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, scratch, nullptr);
  if (st != PA_OK) return st;
  if (num_seqs > 0) {
    // the counters must start at zero; clear them here rather than trust the
    // previous call on this device to have left them so
    if (cudaMemsetAsync(static_cast<char *>(scratch) + ctr_offset, 0, ctr_bytes,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
  }
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, scratch, kStaticScratchBytes,
                   debug_err, stream);
}
