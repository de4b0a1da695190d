// pa_decode_bf16.cu -- decode kernel instantiations for __nv_bfloat16 caches (tensor-core
// path for block sizes that are multiples of 16, CUDA-core path otherwise).
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_SIMT(__nv_bfloat16)
PAGEDKV_INSTANTIATE_MMA(__nv_bfloat16)
PAGEDKV_INSTANTIATE_SHARED(__nv_bfloat16)
PAGEDKV_INSTANTIATE_PREFILL(__nv_bfloat16)
}  // namespace pagedkv
