// pa_decode_inst.cuh -- launcher body shared by the per-dtype translation
// units (each instantiates the decode kernel for one element type, so the
// variants compile in parallel).
#pragma once

#include "pa_decode_impl.cuh"

namespace pagedkv {

template <typename T, int D, int GT>
pa_status launch_decode_partition(const DecodeArgs &a, size_t ring_bytes, cudaStream_t stream) {
  auto kern = decode_partition_kernel<T, D, GT>;
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kRingBytes)) != cudaSuccess)
      return PA_ERR_CUDA;
    configured[dev] = 1;
  }
  kern<<<a.nctas, kDecodeThreads, ring_bytes, stream>>>(a);
  return launch_status();
}

#define PAGEDKV_INSTANTIATE_DECODE(T)                                                            \
  template pa_status launch_decode_partition<T, 64, 1>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_partition<T, 64, 2>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_partition<T, 64, 4>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_partition<T, 64, 8>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_partition<T, 128, 1>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_partition<T, 128, 2>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_partition<T, 128, 4>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_partition<T, 128, 8>(const DecodeArgs &, size_t, cudaStream_t);

}  // namespace pagedkv
