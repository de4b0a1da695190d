// pa_decode.cu -- host entry points of paged decode attention and the
// split-combine kernel (a5).
#include <math.h>

#include "pa_decode_impl.cuh"

namespace pagedkv {

constexpr float kLog2e = 1.4426950408889634f;

// Largest power of two <= 8 dividing the group size: query heads handled by
// one pass over a kv head's blocks.
static int pick_head_chunk(int G) {
  for (int gt = 8; gt > 1; gt >>= 1)
    if (G % gt == 0) return gt;
  return 1;
}

static int decode_grid() { return device_sm_count() * kCtasPerSm; }

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static size_t partial_bytes(int nctas, int head_dim) {
  return round256(size_t(nctas) * 2 * 8 * (head_dim + 2) * sizeof(float));
}

static size_t workspace_bytes_for(int num_seqs, int head_dim, int nctas) {
  return partial_bytes(nctas, head_dim) + round256(size_t(num_seqs + 1) * sizeof(long long));
}

// CTA whose tile range [c*W/N, (c+1)*W/N) holds tile x.
__device__ __forceinline__ int cta_of(long long x, long long W, int N) {
  return int(((x + 1) * N + W - 1) / W - 1);
}

__device__ __forceinline__ long long range_start(int c, long long W, int N) { return (long long)c * W / N; }

template <typename T>
__global__ void __launch_bounds__(128) decode_reduce_kernel(void *out, const int32_t *__restrict__ lens,
                                                            int max_blocks, int S, int Hq, int Hkv, int D, int B,
                                                            int GT, const float *__restrict__ partials,
                                                            const long long *__restrict__ cum, int nctas) {
  const int G = Hq / Hkv;
  const int HC = G / GT;
  const int PC = Hkv * HC;
  const int cap = max_blocks * B;
  const long long W = cum[S];
  for (long long pair = blockIdx.x; pair < (long long)S * PC; pair += gridDim.x) {
    const int s = int(pair / PC);
    const int pc = int(pair - (long long)s * PC);
    const int hq0 = (pc / HC) * G + (pc % HC) * GT;
    int L = lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int nb = (L + B - 1) / B;
    T *o = static_cast<T *>(out) + ((long long)s * Hq + hq0) * D;
    if (nb == 0) {  // nothing cached: zero row
      for (int idx = threadIdx.x; idx < GT * D; idx += blockDim.x) o[idx] = Elem<T>::from_float(0.f);
      continue;
    }
    const long long P0 = cum[s] + (long long)pc * nb;
    const long long P1 = P0 + nb;
    const int cf = cta_of(P0, W, nctas);
    const int cl = cta_of(P1 - 1, W, nctas);
    if (cf == cl) continue;  // finished inside one CTA by the partition kernel
    for (int idx = threadIdx.x; idx < GT * D; idx += blockDim.x) {
      const int h = idx / D;
      const int d = idx - h * D;
      float M = -CUDART_INF_F;
      for (int c = cf; c <= cl; ++c) {
        if (range_start(c, W, nctas) == range_start(c + 1, W, nctas)) continue;
        const int slot = (c == cf && range_start(c, W, nctas) < P0) ? 1 : 0;
        M = fmaxf(M, partials[(((long long)c * 2 + slot) * GT + h) * (D + 2) + D]);
      }
      float num = 0.f, den = 0.f;
      for (int c = cf; c <= cl; ++c) {
        if (range_start(c, W, nctas) == range_start(c + 1, W, nctas)) continue;
        const int slot = (c == cf && range_start(c, W, nctas) < P0) ? 1 : 0;
        const float *rec = partials + (((long long)c * 2 + slot) * GT + h) * (D + 2);
        const float f = fast_exp2(rec[D] - M);
        num += f * rec[d];
        den += f * rec[D + 1];
      }
      o[h * D + d] = Elem<T>::from_float(num / den);
    }
  }
}

struct DecodeShape {
  int G, GT, nctas;
  size_t ring_bytes;
  uint32_t slot_stride;
  int nstage;
};

static pa_status check_decode_args(int max_blocks_per_seq, int num_seqs, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks, pa_dtype dtype,
                                   DecodeShape *shape) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size > kMaxBlockSize) return PA_ERR_UNSUPPORTED;
  if ((long long)max_blocks_per_seq * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  shape->G = num_heads / num_kv_heads;
  shape->GT = pick_head_chunk(shape->G);
  shape->nctas = decode_grid();
  if (shape->nctas <= 0) return PA_ERR_CUDA;
  const size_t slot_bytes = size_t(block_size) * head_dim * dtype_bytes(dtype);
  shape->slot_stride = uint32_t((slot_bytes + 127) & ~size_t(127));
  shape->nstage = int(kRingBytes / shape->slot_stride);
  if (shape->nstage > kMaxStages) shape->nstage = kMaxStages;
  if (shape->nstage < 1) return PA_ERR_UNSUPPORTED;
  shape->ring_bytes = size_t(shape->nstage) * shape->slot_stride;
  return PA_OK;
}

template <typename T>
static pa_status dispatch_partition(const DecodeArgs &a, int D, int GT, size_t ring, cudaStream_t st) {
  if (D == 64) {
    switch (GT) {
      case 1: return launch_decode_partition<T, 64, 1>(a, ring, st);
      case 2: return launch_decode_partition<T, 64, 2>(a, ring, st);
      case 4: return launch_decode_partition<T, 64, 4>(a, ring, st);
      case 8: return launch_decode_partition<T, 64, 8>(a, ring, st);
    }
  } else {
    switch (GT) {
      case 1: return launch_decode_partition<T, 128, 1>(a, ring, st);
      case 2: return launch_decode_partition<T, 128, 2>(a, ring, st);
      case 4: return launch_decode_partition<T, 128, 4>(a, ring, st);
      case 8: return launch_decode_partition<T, 128, 8>(a, ring, st);
    }
  }
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" int pa_decode_grid_size(void) { return decode_grid(); }

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  const int n = decode_grid();
  if (n <= 0) return 0;
  return workspace_bytes_for(num_seqs, head_dim, n);
}

extern "C" pa_status pa_decode_partition(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_seqs, int num_heads,
                                         int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                         float scale, pa_dtype dtype, void *workspace, size_t workspace_bytes,
                                         int *debug_err, void *stream) {
  DecodeShape sh;
  pa_status st = check_decode_args(max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                   num_blocks, dtype, &sh);
  if (st != PA_OK) return st;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(num_seqs, head_dim, sh.nctas)) return PA_ERR_WORKSPACE;

  DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = static_cast<const char *>(k_cache);
  a.v_cache = static_cast<const char *>(v_cache);
  a.tables = block_tables;
  a.lens = context_lens;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.S = num_seqs;
  a.Hq = num_heads;
  a.Hkv = num_kv_heads;
  a.B = block_size;
  a.qscale = scale * kLog2e;
  a.partials = static_cast<float *>(workspace);
  a.cum = reinterpret_cast<long long *>(static_cast<char *>(workspace) + partial_bytes(sh.nctas, head_dim));
  a.err = debug_err;
  a.nctas = sh.nctas;
  a.nstage = sh.nstage;
  a.slot_stride = sh.slot_stride;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case PA_F32: return dispatch_partition<float>(a, head_dim, sh.GT, sh.ring_bytes, s);
    case PA_F16: return dispatch_partition<__half>(a, head_dim, sh.GT, sh.ring_bytes, s);
    case PA_BF16: return dispatch_partition<__nv_bfloat16>(a, head_dim, sh.GT, sh.ring_bytes, s);
  }
  return PA_ERR_INVALID_ARG;
}

extern "C" pa_status pa_decode_reduce(void *out, const int32_t *context_lens, int max_blocks_per_seq, int num_seqs,
                                      int num_heads, int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                                      void *workspace, size_t workspace_bytes, int *debug_err, void *stream) {
  (void)debug_err;
  DecodeShape sh;
  pa_status st = check_decode_args(max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                   1, dtype, &sh);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return PA_OK;
  if (!out || !context_lens || !workspace || !aligned16(out) || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(num_seqs, head_dim, sh.nctas)) return PA_ERR_WORKSPACE;
  const float *partials = static_cast<const float *>(workspace);
  const long long *cum =
      reinterpret_cast<const long long *>(static_cast<const char *>(workspace) + partial_bytes(sh.nctas, head_dim));
  const long long pairs = (long long)num_seqs * num_kv_heads * (sh.G / sh.GT);
  long long grid = pairs;
  const long long cap = (long long)device_sm_count() * 8;
  if (grid > cap) grid = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case PA_F32:
      decode_reduce_kernel<float><<<unsigned(grid), 128, 0, s>>>(out, context_lens, max_blocks_per_seq, num_seqs,
                                                                 num_heads, num_kv_heads, head_dim, block_size,
                                                                 sh.GT, partials, cum, sh.nctas);
      break;
    case PA_F16:
      decode_reduce_kernel<__half><<<unsigned(grid), 128, 0, s>>>(out, context_lens, max_blocks_per_seq, num_seqs,
                                                                  num_heads, num_kv_heads, head_dim, block_size,
                                                                  sh.GT, partials, cum, sh.nctas);
      break;
    case PA_BF16:
      decode_reduce_kernel<__nv_bfloat16><<<unsigned(grid), 128, 0, s>>>(
          out, context_lens, max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, block_size, sh.GT,
          partials, cum, sh.nctas);
      break;
  }
  return launch_status();
}

extern "C" pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, float scale, pa_dtype dtype, void *workspace,
                               size_t workspace_bytes, int *debug_err, void *stream) {
  pa_status st = pa_decode_partition(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                     dtype, workspace, workspace_bytes, debug_err, stream);
  if (st != PA_OK) return st;
  return pa_decode_reduce(out, context_lens, max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim,
                          block_size, dtype, workspace, workspace_bytes, debug_err, stream);
}
