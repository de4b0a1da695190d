// pa_decode_bf16.cu -- decode kernel instantiations for __nv_bfloat16 caches (tensor-core
// path for block sizes that are multiples of 16, CUDA-core path otherwise).
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_SIMT(__nv_bfloat16)
PAGEDKV_INSTANTIATE_MMA(__nv_bfloat16)
PAGEDKV_INSTANTIATE_SHARED(__nv_bfloat16)
PAGEDKV_INSTANTIATE_PREFILL(__nv_bfloat16)
}  // namespace pagedkv

#ifdef PA_TRACE
// Trace builds only (not part of the ABI): copy the bf16 prefill kernel's trace
// arrays out (each translation unit holds its own copy of them).
extern "C" __attribute__((visibility("default"))) int pa_debug_prefill_trace(void *steps, size_t steps_bytes,
                                                                              void *ctas, size_t ctas_bytes) {
  using namespace pagedkv;
  if (steps_bytes > sizeof(pa_prefill_steps_trace) || ctas_bytes > sizeof(pa_prefill_cta_trace)) return -1;
  if (cudaMemcpyFromSymbol(steps, pa_prefill_steps_trace, steps_bytes) != cudaSuccess) return -2;
  if (cudaMemcpyFromSymbol(ctas, pa_prefill_cta_trace, ctas_bytes) != cudaSuccess) return -3;
  return 0;
}
#endif
