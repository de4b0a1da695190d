// pa_decode_f32.cu -- decode kernel instantiations for float elements.
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_DECODE(float)
}  // namespace pagedkv
