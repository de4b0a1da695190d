// pa_kv.cu -- slot lookup, KV write and copy-on-write block copy kernels, the
// write of pa_write_decode, plus the library's shared host helpers.
//
// All four kernels are plain bandwidth kernels: 16-byte vector loads and
// stores, one thread per 16-byte chunk, grid-stride loops over a grid sized
// in multiples of the SM count.

#include "pa_common.cuh"

namespace pagedkv {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Grid for a grid-stride kernel over `work` items: at most a few waves.
static unsigned stride_grid(int64_t work, int threads) {
  const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = int64_t(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

// ----------------------------------------------------------------- a1: slots
__global__ void slot_mapping_kernel(int64_t *__restrict__ slots, const int32_t *__restrict__ tables,
                                    int max_blocks, int num_seqs, const int32_t *__restrict__ token_seq,
                                    const int32_t *__restrict__ token_pos, int64_t n, int B,
                                    int64_t num_blocks, int *err) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int s = token_seq[i];
    const int t = token_pos[i];
    int64_t slot = -1;
    if (t >= 0) {
      const int logical = t / B;
      if (s < 0 || s >= num_seqs || logical >= max_blocks) {
        raise_error(err, PA_DEVERR_POSITION);
      } else {
        const int32_t pid = tables[int64_t(s) * max_blocks + logical];
        if (pid < 0 || pid >= num_blocks)
          raise_error(err, PA_DEVERR_BLOCK_ID);
        else
          slot = int64_t(pid) * B + (t - logical * B);
      }
    }
    slots[i] = slot;
  }
}

// ----------------------------------------------------------------- a2: write
// One thread moves one 16-byte chunk of one (token, head) row of K and of V.
__global__ void write_kv_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                               uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                               const int64_t *__restrict__ slots, int64_t T, int Hkv, int row_chunks, int B,
                               int64_t num_blocks, int *err) {
  const int64_t per_token = int64_t(Hkv) * row_chunks;
  const int64_t total = T * per_token;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tok = i / per_token;
    const int64_t rem = i - tok * per_token;  // head * row_chunks + chunk
    const int64_t slot = slots[tok];
    if (slot < 0) continue;
    if (slot >= num_blocks * B) {
      if (rem == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t pid = slot / B;
    const int64_t off = slot - pid * B;
    const int64_t head = rem / row_chunks;
    const int64_t chunk = rem - head * row_chunks;
    const int64_t dst = ((pid * Hkv + head) * B + off) * row_chunks + chunk;
    k_cache[dst] = key[i];
    v_cache[dst] = value[i];
  }
}

// ----------------------------------------------------------------- a3: COW copy
// blockIdx.y walks the pairs; the x dimension strides over the block's chunks.
__global__ void copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                   const int64_t *__restrict__ pairs, int64_t P, int64_t block_chunks,
                                   int64_t num_blocks, int *err) {
  for (int64_t p = blockIdx.y; p < P; p += gridDim.y) {
    const int64_t src = pairs[2 * p];
    const int64_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4 *ks = k_cache + src * block_chunks;
    const uint4 *vs = v_cache + src * block_chunks;
    uint4 *kd = k_cache + dst * block_chunks;
    uint4 *vd = v_cache + dst * block_chunks;
    for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < block_chunks;
         c += int64_t(gridDim.x) * blockDim.x) {
      const uint4 a = ks[c];
      const uint4 b = vs[c];
      kd[c] = a;
      vd[c] = b;
    }
  }
}

// ------------------------------------------------- a2 for pa_write_decode
// The step's token of each sequence, at position lens[s] - 1, into its slot
// (the lookup of a1 and the write of a2 in one pass): pa_write_decode's write,
// before its decode.  key / value: [S][Hkv][D]; one thread per 16-byte chunk.
__global__ void append_last_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                   uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                   const int32_t *__restrict__ tables, int max_blocks,
                                   const int32_t *__restrict__ lens, int S, int Hkv, int row_chunks, int B,
                                   int64_t num_blocks, int *err) {
  // the decode that follows in pa_write_decode may start launching now: it
  // sets itself up meanwhile and waits for this grid before reading the pools
  launch_dependents();
  const int64_t per_seq = int64_t(Hkv) * row_chunks;
  const int64_t total = int64_t(S) * per_seq;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t s = i / per_seq;
    const int64_t rem = i - s * per_seq;  // head * row_chunks + chunk
    const int L = lens[s];
    if (L <= 0) continue;
    const int t = L - 1;
    const int logical = t / B;
    if (logical >= max_blocks) {
      if (rem == 0) raise_error(err, PA_DEVERR_POSITION);
      continue;
    }
    const int32_t pid = tables[s * max_blocks + logical];
    if (pid < 0 || pid >= num_blocks) {
      if (rem == 0) raise_error(err, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const int64_t head = rem / row_chunks;
    const int64_t chunk = rem - head * row_chunks;
    const int64_t dst = ((int64_t(pid) * Hkv + head) * B + (t - logical * B)) * row_chunks + chunk;
    k_cache[dst] = key[i];
    v_cache[dst] = value[i];
  }
}

pa_status launch_append_last(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int32_t *tables, int max_blocks, const int32_t *lens, int S, int Hkv, int D,
                             int B, int64_t num_blocks, pa_dtype dtype, int *err, cudaStream_t stream) {
  const int row_chunks = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const int64_t work = int64_t(S) * Hkv * row_chunks;
  if (work == 0) return PA_OK;
  const int threads = 256;
  append_last_kernel<<<stride_grid(work, threads), threads, 0, stream>>>(
      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint4 *>(k_cache),
      static_cast<uint4 *>(v_cache), tables, max_blocks, lens, S, Hkv, row_chunks, B, num_blocks, err);
  return launch_status();
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
  }
  return "PA_ERR_UNKNOWN";
}

extern "C" pa_status pa_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables, int max_blocks_per_seq,
                                     int num_seqs, const int32_t *token_seq, const int32_t *token_pos,
                                     int64_t num_tokens, int block_size, int64_t num_blocks, int *debug_err,
                                     void *stream) {
  if (num_tokens < 0 || block_size <= 0 || num_blocks <= 0 || num_seqs < 0 || max_blocks_per_seq < 0)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!slot_mapping || !token_seq || !token_pos || (num_seqs > 0 && max_blocks_per_seq > 0 && !block_tables))
    return PA_ERR_INVALID_ARG;
  const int threads = 256;
  slot_mapping_kernel<<<stride_grid(num_tokens, threads), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      slot_mapping, block_tables, max_blocks_per_seq, num_seqs, token_seq, token_pos, num_tokens, block_size,
      num_blocks, debug_err);
  return launch_status();
}

static bool valid_shape(int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, pa_dtype dtype) {
  if (num_kv_heads <= 0 || block_size <= 0 || block_size > 64 || num_blocks <= 0) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  return dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16;
}

extern "C" pa_status pa_write_kv(const void *key, const void *value, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int64_t num_blocks, pa_dtype dtype, int *debug_err,
                                 void *stream) {
  if (num_tokens < 0 || !valid_shape(num_kv_heads, head_dim, block_size, num_blocks, dtype))
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int row_chunks = static_cast<int>(head_dim * dtype_bytes(dtype) / 16);
  const int64_t work = num_tokens * num_kv_heads * row_chunks;
  const int threads = 256;
  write_kv_kernel<<<stride_grid(work, threads), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint4 *>(k_cache),
      static_cast<uint4 *>(v_cache), slot_mapping, num_tokens, num_kv_heads, row_chunks, block_size, num_blocks,
      debug_err);
  return launch_status();
}

extern "C" pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int64_t num_pairs,
                                    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                    pa_dtype dtype, int *debug_err, void *stream) {
  if (num_pairs < 0 || !valid_shape(num_kv_heads, head_dim, block_size, num_blocks, dtype))
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  const int64_t block_chunks = int64_t(num_kv_heads) * block_size * head_dim * dtype_bytes(dtype) / 16;
  const int threads = 256;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
  // enough CTAs in flight: ~4 per SM overall, split between pairs and chunks
  int64_t gy = num_pairs < 65535 ? num_pairs : 65535;
  int64_t gx = (int64_t(sms) * 4 + gy - 1) / gy;
  const int64_t gx_max = (block_chunks + threads - 1) / threads;
  if (gx > gx_max) gx = gx_max;
  if (gx < 1) gx = 1;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  copy_blocks_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs, num_pairs, block_chunks, num_blocks,
      debug_err);
  return launch_status();
}
