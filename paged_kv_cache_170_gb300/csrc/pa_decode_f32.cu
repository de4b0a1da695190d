// pa_decode_f32.cu -- decode kernel instantiations for fp32 caches (CUDA-core path).
#include "pa_decode_inst.cuh"

namespace pagedkv {
PAGEDKV_INSTANTIATE_SIMT(float)
}  // namespace pagedkv
