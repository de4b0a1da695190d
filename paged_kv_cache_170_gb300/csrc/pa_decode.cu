// pa_decode.cu -- host entry points of paged decode attention and the choice
// between the tensor-core and CUDA-core kernels.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "pa_decode_shared.cuh"
#include "pa_prefill.cuh"
#include "pa_sched.cuh"

namespace pagedkv {

template <typename T, int D, int GT>
pa_status launch_decode_simt(const DecodeArgs &a, size_t ring_bytes, cudaStream_t stream);
template <typename T, int D>
pa_status launch_decode_mma(const DecodeArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t ring_bytes,
                            cudaStream_t stream, bool early);
template <typename T, int D>
pa_status launch_decode_shared(const SharedArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t ring_bytes,
                               cudaStream_t stream, bool early);
template <typename T, int D>
pa_status launch_merge_shared(const MergeArgs &a, cudaStream_t stream);
template <typename T, int D, bool kGroups>
pa_status launch_prefill(const PrefillArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, size_t smem_bytes,
                            dim3 grid, cudaStream_t stream);

pa_status launch_append_last(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int32_t *tables, int max_blocks, const int32_t *lens, int S, int Hkv, int D,
                             int B, int64_t num_blocks, pa_dtype dtype, int *err, cudaStream_t stream);

constexpr float kLog2e = 1.4426950408889634f;

static int decode_grid() { return device_sm_count() * kCtasPerSm; }

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Two partial records per CTA, sized for the largest head_dim whatever the
// call's: the counters that follow then start at the same offset for every
// call on this device, so calls of any shapes can share one workspace
// without one call's records landing on another call's counters.
static size_t partial_bytes(int nctas, int head_dim) {
  (void)head_dim;
  return round256(size_t(nctas) * 2 * 8 * state_row(128) * sizeof(float));
}

// partial records, then one counter per (sequence, query head) (an upper
// bound of the split pairs)
static size_t workspace_bytes_for(int num_seqs, int num_heads, int head_dim, int nctas) {
  return partial_bytes(nctas, head_dim) + round256(size_t(num_seqs) * num_heads * sizeof(unsigned));
}

bool decode_counter_region(int num_seqs, int num_heads, int head_dim, size_t *offset, size_t *bytes) {
  const int n = decode_grid();
  if (n <= 0 || num_seqs < 0 || num_heads <= 0 || (head_dim != 64 && head_dim != 128)) return false;
  *offset = partial_bytes(n, head_dim);
  *bytes = size_t(num_seqs) * num_heads * sizeof(unsigned);
  return true;
}

// ----------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A pool [NB][Hkv][B][D] seen as NB*Hkv*B rows of D 16-bit elements, loaded
// with the 128-byte swizzle into [D/64 halves][B rows][128 bytes].  With
// three_d (D = 128) the map is (64 elements, rows, 2 halves) with the halves
// 128 bytes apart, so one box {64, B, 2} brings a whole tile; otherwise one
// 2-D box {64, B} per half.
static bool encode_pool_map(CUtensorMap *map, const void *pool, pa_dtype dtype, int64_t num_blocks, int Hkv,
                            int B, int D, bool three_d) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const CUtensorMapDataType ty =
      dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t rows = cuuint64_t(num_blocks) * Hkv * B;
  if (three_d) {
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, 128};
    const cuuint32_t box[3] = {64, cuuint32_t(B), 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, ty, 3, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[2] = {cuuint64_t(D), rows};
  const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(B)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, ty, 2, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ----------------------------------------------------------------- dispatch
struct DecodeShape {
  int G, GT, nctas;
  bool mma;
  size_t ring_bytes;
  uint32_t slot_stride, tile_stride, q_offset, q_bytes;
  int nstage, ncw, pg;
};

// Largest power of two <= 8 dividing G (CUDA-core kernel, GT is a template
// parameter there) or largest divisor <= 8 (tensor-core kernel, which covers
// up to 8 heads with one N = 8 MMA tile).
static int pick_head_chunk(int G, bool mma) {
  if (mma) {
    for (int gt = 8; gt > 1; --gt)
      if (G % gt == 0) return gt;
    return 1;
  }
  for (int gt = 8; gt > 1; gt >>= 1)
    if (G % gt == 0) return gt;
  return 1;
}

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
  if (num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  shape->G = num_heads / num_kv_heads;
  shape->mma = dtype != PA_F32 && block_size % 16 == 0 && tensor_map_encoder() != nullptr;
  shape->GT = pick_head_chunk(shape->G, shape->mma);
  shape->nctas = decode_grid();
  if (shape->nctas <= 0) return PA_ERR_CUDA;
  // one ring slot holds the K tile and the V tile of one (block, kv head);
  // on the tensor-core path also room for the q rows of one pair chunk
  const size_t tile_bytes = size_t(block_size) * head_dim * dtype_bytes(dtype);
  const size_t align = shape->mma ? 1024 : 128;  // the swizzled tiles repeat every 1024 bytes
  shape->tile_stride = uint32_t((tile_bytes + align - 1) / align * align);
  shape->q_offset = 2 * shape->tile_stride;
  shape->q_bytes = shape->mma ? uint32_t(shape->GT * head_dim * dtype_bytes(dtype)) : 0u;
  shape->slot_stride = uint32_t((shape->q_offset + shape->q_bytes + align - 1) / align * align);
  shape->nstage = int((shape->mma ? kRingBytesMma : kRingBytes) / shape->slot_stride);
  if (shape->nstage > kMaxStages) shape->nstage = kMaxStages;
  if (shape->nstage < 1) return PA_ERR_UNSUPPORTED;
  // consumer warps and producer group size with ncw + pg <= nstage (the ring's
  // phase argument needs it; see wait_entry): keep 4 consumers when the ring
  // allows and give the producer what is left, up to 4 entries at a time
  shape->ncw = shape->nstage - 1 < kConsumerWarps ? (shape->nstage > 1 ? shape->nstage - 1 : 1) : kConsumerWarps;
  shape->pg = shape->nstage - shape->ncw;
  if (shape->pg > 4) shape->pg = 4;
  if (shape->pg < 1) shape->pg = 1;
  shape->ring_bytes = size_t(shape->nstage) * shape->slot_stride;
  return PA_OK;
}

template <typename T>
static pa_status dispatch_simt(const DecodeArgs &a, int D, int GT, size_t ring, cudaStream_t st) {
  if (D == 64) {
    switch (GT) {
      case 1: return launch_decode_simt<T, 64, 1>(a, ring, st);
      case 2: return launch_decode_simt<T, 64, 2>(a, ring, st);
      case 4: return launch_decode_simt<T, 64, 4>(a, ring, st);
      case 8: return launch_decode_simt<T, 64, 8>(a, ring, st);
    }
  } else {
    switch (GT) {
      case 1: return launch_decode_simt<T, 128, 1>(a, ring, st);
      case 2: return launch_decode_simt<T, 128, 2>(a, ring, st);
      case 4: return launch_decode_simt<T, 128, 4>(a, ring, st);
      case 8: return launch_decode_simt<T, 128, 8>(a, ring, st);
    }
  }
  return PA_ERR_UNSUPPORTED;
}

// Tensor maps of the K and V pools: one 3-D box per tile when the encoder
// takes the (rows, halves) stride order, else one 2-D box per 64-column half
// (*nops = copies per tile; D = 64 is always one 2-D box).
static bool encode_pool_maps(const void *k_cache, const void *v_cache, pa_dtype dtype, int64_t num_blocks, int Hkv,
                             int B, int D, CUtensorMap *mk, CUtensorMap *mv, int *nops) {
  *nops = 1;
  if (D == 128 && encode_pool_map(mk, k_cache, dtype, num_blocks, Hkv, B, D, true) &&
      encode_pool_map(mv, v_cache, dtype, num_blocks, Hkv, B, D, true))
    return true;
  if (!encode_pool_map(mk, k_cache, dtype, num_blocks, Hkv, B, D, false) ||
      !encode_pool_map(mv, v_cache, dtype, num_blocks, Hkv, B, D, false))
    return false;
  *nops = D == 64 ? 1 : 2;
  return true;
}

template <typename T>
static pa_status dispatch_mma(const DecodeArgs &a, const void *k_cache, const void *v_cache, pa_dtype dtype, int D,
                              size_t ring, cudaStream_t st, bool early = false) {
  CUtensorMap mk, mv;
  DecodeArgs b = a;
  if (!encode_pool_maps(k_cache, v_cache, dtype, a.num_blocks, a.Hkv, a.B, D, &mk, &mv, &b.nops)) return PA_ERR_CUDA;
  return D == 64 ? launch_decode_mma<T, 64>(b, mk, mv, ring, st, early)
                 : launch_decode_mma<T, 128>(b, mk, mv, ring, st, early);
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" int pa_decode_grid_size(void) { return decode_grid(); }

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  const int n = decode_grid();
  if (n <= 0) return 0;
  return workspace_bytes_for(num_seqs, num_heads, head_dim, n);
}

namespace pagedkv {

// The host-side checks of a decode call (everything but the workspace size):
// PA_OK when pa_decode would go on to launch (or, for num_seqs == 0, return
// PA_OK without work).
pa_status check_decode_call(const void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, float scale, pa_dtype dtype, const void *workspace,
                            DecodeShape *shape) {
  DecodeShape local;
  DecodeShape &sh = shape != nullptr ? *shape : local;
  const pa_status st = check_decode_args(max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim,
                                         block_size, num_blocks, dtype, &sh);
  if (st != PA_OK) return st;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// pa_decode, or (new_key non-null, pa_write_decode) with each sequence's
// token at position context_lens[s] - 1 written first.  early_launch: the
// previous kernel in the stream lets this one start launching before it ends
// (it triggers griddepcontrol.launch_dependents); the decode's producer waits
// for it before its first copy.
static pa_status decode_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, float scale, pa_dtype dtype, void *workspace, size_t workspace_bytes,
                             int *debug_err, void *stream, const void *new_key = nullptr,
                             const void *new_value = nullptr,
                             bool early_launch = false) {
  DecodeShape sh;
  pa_status st = check_decode_call(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                   num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                                   workspace, &sh);
  if (st != PA_OK || num_seqs == 0) return st;
  if (workspace_bytes < workspace_bytes_for(num_seqs, num_heads, head_dim, sh.nctas)) return PA_ERR_WORKSPACE;
  if (new_key != nullptr && (new_value == nullptr || !aligned16(new_key) || !aligned16(new_value)))
    return PA_ERR_INVALID_ARG;

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
  a.counters = reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + partial_bytes(sh.nctas, head_dim));
  a.err = debug_err;
  a.nctas = sh.nctas;
  a.nstage = sh.nstage;
  a.slot_stride = sh.slot_stride;
  a.tile_stride = sh.tile_stride;
  a.GT = sh.GT;
  a.ncw = sh.ncw;
  a.pg = sh.pg;
  a.nops = 1;
  a.q_offset = sh.q_offset;
  a.q_bytes = sh.q_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool early = early_launch && sh.mma;  // the decode may start launching while the previous kernel runs
  if (new_key != nullptr) {
    const pa_status w = launch_append_last(new_key, new_value, const_cast<void *>(k_cache),
                                           const_cast<void *>(v_cache), block_tables, max_blocks_per_seq,
                                           context_lens, num_seqs, num_kv_heads, head_dim, block_size, num_blocks,
                                           dtype, debug_err, s);
    if (w != PA_OK) return w;
    early = sh.mma;
  }
  if (sh.mma) {
    return dtype == PA_BF16
               ? dispatch_mma<__nv_bfloat16>(a, k_cache, v_cache, dtype, head_dim, sh.ring_bytes, s, early)
               : dispatch_mma<__half>(a, k_cache, v_cache, dtype, head_dim, sh.ring_bytes, s, early);
  }
  switch (dtype) {
    case PA_F32: return dispatch_simt<float>(a, head_dim, sh.GT, sh.ring_bytes, s);
    case PA_F16: return dispatch_simt<__half>(a, head_dim, sh.GT, sh.ring_bytes, s);
    case PA_BF16: return dispatch_simt<__nv_bfloat16>(a, head_dim, sh.GT, sh.ring_bytes, s);
  }
  return PA_ERR_INVALID_ARG;
}

}  // namespace pagedkv

extern "C" pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, float scale, pa_dtype dtype, void *workspace,
                               size_t workspace_bytes, int *debug_err, void *stream) {
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace, workspace_bytes,
                     debug_err, stream);
}

extern "C" pa_status pa_write_decode(void *out, const void *q, const void *new_key, const void *new_value,
                                     void *k_cache, void *v_cache, const int32_t *block_tables,
                                     int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                     int num_heads, int num_kv_heads, int head_dim, int block_size,
                                     int64_t num_blocks, float scale, pa_dtype dtype, void *workspace,
                                     size_t workspace_bytes, int *debug_err, void *stream) {
  if (num_seqs > 0 && (new_key == nullptr || new_value == nullptr)) return PA_ERR_INVALID_ARG;
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace, workspace_bytes,
                     debug_err, stream, new_key, new_value);
}

// ------------------------------------------------------ shared-block decode
namespace pagedkv {

// The plan's header if it belongs to these arguments, else null.
static const SharePlanHeader *check_plan(const int32_t *plan_host, int num_seqs, int num_heads, int num_kv_heads,
                                         int block_size, int max_blocks_per_seq) {
  if (plan_host == nullptr) return nullptr;
  const SharePlanHeader *h = reinterpret_cast<const SharePlanHeader *>(plan_host);
  if (h->magic != kSharePlanMagic || h->num_seqs != num_seqs || num_kv_heads <= 0 ||
      h->group_size * num_kv_heads != num_heads || h->num_kv_heads != num_kv_heads || h->block_size != block_size ||
      h->max_blocks != max_blocks_per_seq || h->nctas <= 0 || h->num_pieces < 0 || h->total_ints < kSharePlanHeaderInts ||
      h->num_shared_groups < 0 || h->num_shared_groups > h->num_groups || (h->p_desc & 3) != 0 ||
      h->num_tc_items < 0 || (h->t_items & 3) != 0 ||
      (long long)h->t_items + (long long)h->num_tc_items * kTcItemInts > h->total_ints || h->t_qrow < 0 ||
      (long long)h->t_qrow + (long long)h->num_tc_items * kTcItemRows > h->total_ints || h->t_blk < 0 ||
      h->t_blk_stride < 0 || (long long)h->t_blk + (long long)h->num_tc_items * h->t_blk_stride > h->total_ints ||
      (long long)h->r_off + (long long)num_seqs * num_heads + 1 > h->total_ints || h->r_rec > h->total_ints)
    return nullptr;
  return h;
}

// Workspace of the shared-block decode: the step-1 kernel's partial states
// [num_pieces][kSharePassRows][state_row(D)]; for a plan with no shared group
// (the call is then pa_decode), pa_decode's workspace.
static size_t shared_workspace_bytes(const SharePlanHeader &h, int num_seqs, int num_heads, int head_dim,
                                     int nctas) {
  if (h.num_shared_groups == 0) return workspace_bytes_for(num_seqs, num_heads, head_dim, nctas);
  return round256(size_t(h.num_pieces) * kSharePassRows * state_row(head_dim) * sizeof(float));
}

template <typename T>
static pa_status shared_step(const SharedArgs &sa, const void *k_cache, const void *v_cache, pa_dtype dtype, int D,
                             size_t ring, cudaStream_t st, bool early) {
  CUtensorMap mk, mv;
  SharedArgs b = sa;
  if (!encode_pool_maps(k_cache, v_cache, dtype, sa.num_blocks, sa.Hkv, sa.B, D, &mk, &mv, &b.nops))
    return PA_ERR_CUDA;
  return D == 64 ? launch_decode_shared<T, 64>(b, mk, mv, ring, st, early)
                 : launch_decode_shared<T, 128>(b, mk, mv, ring, st, early);
}

template <typename T, bool kGroups = false>
static pa_status prefill_dispatch(const PrefillArgs &pa_args, const void *k_cache, const void *v_cache,
                                  pa_dtype dtype, int D, size_t smem, dim3 grid, cudaStream_t st) {
  CUtensorMap mk, mv;
  PrefillArgs b = pa_args;
  // K: one 2-D box (B rows x 64 columns) per block and half; V: one box per
  // block (a 3-D box over both halves when head_dim is 128)
  if (!encode_pool_map(&mk, k_cache, dtype, b.num_blocks, b.Hkv, b.B, D, false) ||
      !encode_pool_map(&mv, v_cache, dtype, b.num_blocks, b.Hkv, b.B, D, D == 128))
    return PA_ERR_CUDA;
  return D == 64 ? launch_prefill<T, 64, kGroups>(b, mk, mv, smem, grid, st)
                 : launch_prefill<T, 128, kGroups>(b, mk, mv, smem, grid, st);
}

template <typename T>
static pa_status merge_step(const MergeArgs &ma, int D, cudaStream_t st) {
  return D == 64 ? launch_merge_shared<T, 64>(ma, st) : launch_merge_shared<T, 128>(ma, st);
}

}  // namespace pagedkv

extern "C" size_t pa_decode_shared_workspace_size(const int32_t *plan_host, int num_seqs, int num_heads,
                                                  int num_kv_heads, int head_dim) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  const SharePlanHeader *h = reinterpret_cast<const SharePlanHeader *>(plan_host);
  if (h == nullptr || h->magic != kSharePlanMagic || h->num_seqs != num_seqs) return 0;
  const int n = decode_grid();
  if (n <= 0) return 0;
  return shared_workspace_bytes(*h, num_seqs, num_heads, head_dim, n);
}

extern "C" pa_status pa_decode_shared(void *out, const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int64_t num_blocks, float scale, pa_dtype dtype,
                                      const int32_t *plan_host, const int32_t *plan_dev, void *workspace,
                                      size_t workspace_bytes, int *debug_err, void *stream) {
  DecodeShape sh;
  pa_status st = check_decode_args(max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                   num_blocks, dtype, &sh);
  if (st != PA_OK) return st;
  if (!sh.mma) return PA_ERR_UNSUPPORTED;  // fp16 / bf16 with block_size % 16 == 0 only
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  const SharePlanHeader *h =
      check_plan(plan_host, num_seqs, num_heads, num_kv_heads, block_size, max_blocks_per_seq);
  if (h == nullptr) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (h->num_shared_groups == 0)  // nothing shared: the plain decode
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace, workspace_bytes,
                     debug_err, stream);
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace || !plan_dev)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace) ||
      !aligned16(plan_dev))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < shared_workspace_bytes(*h, num_seqs, num_heads, head_dim, sh.nctas)) return PA_ERR_WORKSPACE;
  float *records = static_cast<float *>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // 1. every group's blocks: the shared runs once per group of sharers, and
  // each sequence's own blocks
  SharedArgs sa;
  sa.q = q;
  sa.tables = block_tables;
  sa.lens = context_lens;
  sa.plan = plan_dev;
  sa.h = *h;
  sa.num_blocks = num_blocks;
  sa.max_blocks = max_blocks_per_seq;
  sa.S = num_seqs;
  sa.Hq = num_heads;
  sa.Hkv = num_kv_heads;
  sa.B = block_size;
  sa.qscale = scale * kLog2e;
  sa.records = records;
  sa.err = debug_err;
  sa.tile_stride = sh.tile_stride;
  sa.slot_stride = 2 * sh.tile_stride;
  sa.nstage = int(kRingBytesShared / sa.slot_stride);
  if (sa.nstage > kMaxStages) sa.nstage = kMaxStages;
  if (sa.nstage < 1) return PA_ERR_UNSUPPORTED;
  sa.pg = sa.nstage < 4 ? sa.nstage : 4;
  sa.nops = 1;
  const size_t ring = size_t(sa.nstage) * sa.slot_stride;
  MergeArgs ma;
  ma.out = out;
  ma.records = records;
  ma.plan = plan_dev;
  ma.h = *h;
  ma.S = num_seqs;
  ma.Hq = num_heads;
  // 1a. the groups with many sharers, on the tensor cores (one CTA per item)
  if (h->num_tc_items > 0) {
    if (block_size % 16 != 0 || kTcStepTokens % block_size != 0) return PA_ERR_INVALID_ARG;  // no such plan
    PrefillArgs ta;
    memset(&ta, 0, sizeof(ta));
    ta.q = q;
    ta.tables = block_tables;
    ta.lens = context_lens;
    ta.num_blocks = num_blocks;
    ta.max_blocks = max_blocks_per_seq;
    ta.S = num_seqs;
    ta.Hq = num_heads;
    ta.Hkv = num_kv_heads;
    ta.B = block_size;
    ta.qscale = scale * kLog2e;
    ta.err = debug_err;
    ta.records = records;
    ta.plan = plan_dev;
    ta.t_items = h->t_items;
    ta.t_qrow = h->t_qrow;
    ta.t_blk = h->t_blk;
    ta.t_blk_stride = h->t_blk_stride;
    const size_t smem = size_t(tc_smem_bytes(head_dim));
    const dim3 grid{unsigned(h->num_tc_items), 1u, 1u};
    st = dtype == PA_BF16 ? prefill_dispatch<__nv_bfloat16, true>(ta, k_cache, v_cache, dtype, head_dim, smem, grid, s)
                          : prefill_dispatch<__half, true>(ta, k_cache, v_cache, dtype, head_dim, smem, grid, s);
    if (st != PA_OK) return st;
  }
  // 1b. every other group's blocks, in the CTAs' pieces; launched early
  // beside 1a (it reads nothing 1a writes), so its CTAs fill the SMs 1a
  // leaves idle
  const long long mma_pieces = (long long)plan_host[h->c_poff + h->nctas] - plan_host[h->c_poff] +
                               plan_host[h->c_opoff + h->nctas] - plan_host[h->c_opoff];
  if (mma_pieces > 0) {
    const bool early = h->num_tc_items > 0;
    st = dtype == PA_BF16 ? shared_step<__nv_bfloat16>(sa, k_cache, v_cache, dtype, head_dim, ring, s, early)
                          : shared_step<__half>(sa, k_cache, v_cache, dtype, head_dim, ring, s, early);
    if (st != PA_OK) return st;
  }
  // 2. merge
  return dtype == PA_BF16 ? merge_step<__nv_bfloat16>(ma, head_dim, s) : merge_step<__half>(ma, head_dim, s);
}

// ------------------------------------------------------------------ prefill

extern "C" pa_status pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                                const int32_t *q_start, int num_seqs, int max_q_len, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                                pa_dtype dtype, int *debug_err, void *stream) {
  if (num_seqs < 0 || max_q_len < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || !isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  // a block must be an MMA column group (16 tokens) and divide the 64-token softmax step
  if (dtype == PA_F32 || block_size % 16 != 0 || kTcStepTokens % block_size != 0) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if ((long long)max_blocks_per_seq * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (tensor_map_encoder() == nullptr) return PA_ERR_UNSUPPORTED;
  const long long tiles = ((long long)max_q_len * (num_heads / num_kv_heads) + kTcRows - 1) / kTcRows;
  if (num_seqs == 0 || tiles == 0) return PA_OK;
  if (tiles * num_seqs * num_kv_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !q_start) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;

  PrefillArgs a;
  a.out = out;
  a.q = q;
  a.tables = block_tables;
  a.lens = context_lens;
  a.q_start = q_start;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.S = num_seqs;
  a.Hq = num_heads;
  a.Hkv = num_kv_heads;
  a.B = block_size;
  a.qscale = scale * kLog2e;
  a.err = debug_err;
  // dynamic shared memory: the Q tile and the K and V rings, no slack (the
  // kernel checks the 1024-byte alignment its swizzled tiles need)
  const size_t smem = size_t(tc_smem_bytes(head_dim));
  const dim3 grid{unsigned(tiles * num_seqs * num_kv_heads), 1u, 1u};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dtype == PA_BF16 ? prefill_dispatch<__nv_bfloat16>(a, k_cache, v_cache, dtype, head_dim, smem, grid, s)
                          : prefill_dispatch<__half>(a, k_cache, v_cache, dtype, head_dim, smem, grid, s);
}
