// pa_decode_f16.cu -- decode kernel instantiations for __half caches (tensor-core
// path for block sizes that are multiples of 16, CUDA-core path otherwise).
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_SIMT(__half)
PAGEDKV_INSTANTIATE_MMA(__half)
PAGEDKV_INSTANTIATE_SHARED(__half)
PAGEDKV_INSTANTIATE_PREFILL(__half)
}  // namespace pagedkv
