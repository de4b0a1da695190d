// pa_decode_f16.cu -- decode kernel instantiations for __half elements.
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_DECODE(__half)
}  // namespace pagedkv
