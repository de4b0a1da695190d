// pa_decode_inst.cuh -- launchers shared by the per-dtype translation units
// (each instantiates the decode kernels for one element type, so the variants
// compile in parallel).
#pragma once

#include "pa_decode_mma.cuh"
#include "pa_decode_shared.cuh"
#include "pa_decode_simt.cuh"
#include "pa_prefill.cuh"

namespace pagedkv {

// Opt a kernel in to the ring's dynamic shared memory once per device.
template <typename K>
inline bool configure_once(K kern, int bytes, int *configured) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    configured[dev] = 1;
  }
  return true;
}

template <typename T, int D, int GT>
pa_status launch_decode_simt(const DecodeArgs &a, size_t ring_bytes, cudaStream_t stream) {
  static int configured[64] = {0};
  auto kern = decode_partition_kernel<T, D, GT>;
  if (!configure_once(kern, kRingBytes, configured)) return PA_ERR_CUDA;
  kern<<<a.nctas, kDecodeThreads, ring_bytes, stream>>>(a);
  return launch_status();
}

// early: allow the launch to start while the previous kernel in the stream
// is still running (programmatic dependent launch); the kernel's producer
// waits for that kernel before its first copy from the pools.
template <typename T, int D>
pa_status launch_decode_mma(const DecodeArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t ring_bytes,
                            cudaStream_t stream, bool early) {
  static int configured[64] = {0};
  auto kern = decode_partition_mma_kernel<T, D>;
  if (!configure_once(kern, kRingBytesMma + 1024, configured)) return PA_ERR_CUDA;
  if (!early) {
    kern<<<a.nctas, kDecodeThreads, ring_bytes + 1024, stream>>>(a, mk, mv);
    return launch_status();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nctas);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = ring_bytes + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a, mk, mv) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return launch_status();
}

// early: may start while the previous kernel (the tensor-core groups') runs.
template <typename T, int D>
pa_status launch_decode_shared(const SharedArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t ring_bytes,
                               cudaStream_t stream, bool early) {
  static int configured[64] = {0};
  auto kern = decode_shared_mma_kernel<T, D>;
  if (!configure_once(kern, kRingBytesShared + 1024, configured)) return PA_ERR_CUDA;
  if (!early) {
    kern<<<a.h.nctas, kSharedThreads, ring_bytes + 1024, stream>>>(a, mk, mv);
    return launch_status();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.h.nctas);
  cfg.blockDim = dim3(kSharedThreads);
  cfg.dynamicSmemBytes = ring_bytes + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a, mk, mv) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return launch_status();
}

template <typename T, int D>
pa_status launch_merge_shared(const MergeArgs &a, cudaStream_t stream) {
  const long long rows = (long long)a.S * a.Hq;
  if (rows == 0) return PA_OK;
  merge_shared_kernel<T, D><<<unsigned((rows + kMergeWarps - 1) / kMergeWarps), kMergeWarps * 32, 0, stream>>>(a);
  return launch_status();
}

// kGroups: the shared-block decode's dense groups (grid = the plan's items).
template <typename T, int D, bool kGroups>
pa_status launch_prefill(const PrefillArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t smem_bytes,
                            dim3 grid, cudaStream_t stream) {
  static int configured[64] = {0};
  auto kern = prefill_tc_kernel<T, D, kGroups>;
  if (!configure_once(kern, tc_smem_bytes(D), configured)) return PA_ERR_CUDA;
  kern<<<grid, kTcThreads, smem_bytes, stream>>>(a, mk, mv);
  return launch_status();
}

#define PAGEDKV_INSTANTIATE_PREFILL(T)                                                                           \
  template pa_status launch_prefill<T, 64, false>(const PrefillArgs &, const CUtensorMap &, const CUtensorMap &, \
                                                  size_t, dim3, cudaStream_t);                                   \
  template pa_status launch_prefill<T, 128, false>(const PrefillArgs &, const CUtensorMap &,                     \
                                                   const CUtensorMap &, size_t, dim3, cudaStream_t);             \
  template pa_status launch_prefill<T, 64, true>(const PrefillArgs &, const CUtensorMap &, const CUtensorMap &,  \
                                                 size_t, dim3, cudaStream_t);                                    \
  template pa_status launch_prefill<T, 128, true>(const PrefillArgs &, const CUtensorMap &, const CUtensorMap &, \
                                                  size_t, dim3, cudaStream_t);

#define PAGEDKV_INSTANTIATE_SHARED(T)                                                                         \
  template pa_status launch_decode_shared<T, 64>(const SharedArgs &, const CUtensorMap &, const CUtensorMap &, \
                                                 size_t, cudaStream_t, bool);                                  \
  template pa_status launch_decode_shared<T, 128>(const SharedArgs &, const CUtensorMap &,                     \
                                                  const CUtensorMap &, size_t, cudaStream_t, bool);            \
  template pa_status launch_merge_shared<T, 64>(const MergeArgs &, cudaStream_t);                              \
  template pa_status launch_merge_shared<T, 128>(const MergeArgs &, cudaStream_t);

#define PAGEDKV_INSTANTIATE_SIMT(T)                                                           \
  template pa_status launch_decode_simt<T, 64, 1>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_simt<T, 64, 2>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_simt<T, 64, 4>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_simt<T, 64, 8>(const DecodeArgs &, size_t, cudaStream_t);  \
  template pa_status launch_decode_simt<T, 128, 1>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_simt<T, 128, 2>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_simt<T, 128, 4>(const DecodeArgs &, size_t, cudaStream_t); \
  template pa_status launch_decode_simt<T, 128, 8>(const DecodeArgs &, size_t, cudaStream_t);

#define PAGEDKV_INSTANTIATE_MMA(T)                                                                          \
  template pa_status launch_decode_mma<T, 64>(const DecodeArgs &, const CUtensorMap &, const CUtensorMap &, \
                                              size_t, cudaStream_t, bool);                                  \
  template pa_status launch_decode_mma<T, 128>(const DecodeArgs &, const CUtensorMap &, const CUtensorMap &, \
                                               size_t, cudaStream_t, bool);

}  // namespace pagedkv
