// pa_decode_bf16.cu -- decode kernel instantiations for __nv_bfloat16 elements.
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_DECODE(__nv_bfloat16)
}  // namespace pagedkv
