/*
 * pagedkv.h -- C ABI of libpagedkv.so: paged KV-cache decode attention on
 * NVIDIA GB300 (sm_103a).
 *
 * The KV cache is split into fixed-size physical blocks of B tokens; each
 * sequence owns a block table mapping its logical block i to a physical block
 * id, so token position t lives in physical block block_table[t / B] at
 * offset t % B (aiqz.cc "paged-attention-mechanism", section "块表映射机制";
 * lihaoran.work "auto-20261007-1900", section "块表把逻辑顺序映射到物理位置").
 *
 * Layouts (row-major, element type given by pa_dtype):
 *   q, out            [S][Hq][D]
 *   k_cache, v_cache  [NB][Hkv][B][D]   one (block, kv head) tile is B*D
 *                                        contiguous elements
 *   block_tables      int32 [S][max_blocks_per_seq]; entries past
 *                     ceil(context_len / B) are never read (may hold -1)
 *   context_lens      int32 [S]
 *   slot_mapping      int64 [T]; slot = pid * B + offset, slot < 0 = skip
 *
 * Conventions for every call:
 *   - All pointers are device pointers owned by the caller (allocated by the
 *     caller, e.g. through PyTorch).  Calls never allocate, never free and
 *     never synchronise: they enqueue kernels on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and return.
 *   - Host-side scalar arguments are validated; a bad one returns
 *     PA_ERR_INVALID_ARG (or PA_ERR_UNSUPPORTED for a valid but unsupported
 *     shape) and enqueues nothing.  A failed launch returns PA_ERR_CUDA.
 *   - Device-side data (table entries, slots, lengths) is range-checked in the
 *     kernels: an offending access is skipped and a bit is OR-ed into
 *     *debug_err (a caller-owned device int; may be NULL to ignore).  Results
 *     touched by a skipped access are unspecified.  The bits are PA_DEVERR_*.
 *   - Device pointers must be 16-byte aligned; head_dim must be 64 or 128;
 *     block_size in [1, 64]; num_heads a multiple of num_kv_heads.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are exported even when the library hides everything else. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,
  PA_ERR_UNSUPPORTED = 2,
  PA_ERR_CUDA = 3,
  PA_ERR_WORKSPACE = 4
} pa_status;

/* Bits OR-ed into *debug_err by the kernels. */
#define PA_DEVERR_BLOCK_ID 1u  /* a block id outside [0, num_blocks)          */
#define PA_DEVERR_SLOT 2u      /* a slot >= num_blocks * block_size           */
#define PA_DEVERR_CONTEXT 4u   /* context_len < 0 or > max_blocks_per_seq * B */
#define PA_DEVERR_TIMEOUT 8u   /* an internal pipeline wait gave up (~1.5 s)  */
#define PA_DEVERR_POSITION 16u /* a token position outside its block table    */
#define PA_DEVERR_LAYOUT 32u   /* shared memory not 1024-byte aligned (internal; the launch did no work) */

/* Human-readable name of a status code (static string). */
PA_API const char *pa_status_string(pa_status status);

/*
 * a1 -- slot of each new token (the host-side "append" emits it; this is the
 * same lookup on the device).  Token i belongs to sequence token_seq[i] at
 * position token_pos[i]:
 *     slot_mapping[i] = block_tables[seq][pos / B] * B + pos % B
 * (aiqz.cc, section "块表映射机制").  A negative position gives slot -1
 * (padding).  A sequence index outside [0, num_seqs), a position past the
 * table row, or a block id outside [0, num_blocks) gives slot -1 and sets a
 * PA_DEVERR bit.
 */
PA_API pa_status pa_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                          int max_blocks_per_seq, int num_seqs,
                          const int32_t *token_seq, const int32_t *token_pos,
                          int64_t num_tokens, int block_size, int64_t num_blocks,
                          int *debug_err, void *stream);

/*
 * a2 -- write each new token's K and V rows into its slot (bit copy):
 *     k_cache[slot / B][h][slot % B][:] = key[i][h][:]   (same for V)
 * for every token i and kv head h; slot < 0 skips the token (padding).
 * Writing the new token is the last step of an append or of a copy-on-write
 * (aiqz.cc, section "前缀共享机制").  key/value: [T][Hkv][D].  Slots must be
 * unique within one call.
 */
PA_API pa_status pa_write_kv(const void *key, const void *value, void *k_cache,
                      void *v_cache, const int64_t *slot_mapping,
                      int64_t num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int64_t num_blocks, pa_dtype dtype,
                      int *debug_err, void *stream);

/*
 * a3 -- copy-on-write block copy: for each pair p, the whole physical block
 * pairs[p][1] (dst) of K and of V, all heads and all B slots, becomes a copy
 * of block pairs[p][0] (src) (aiqz.cc, section "前缀共享机制"; cf-1.com
 * news/5879632, section 4.2).  pairs: device int64 [P][2].  Within one call
 * every dst must be distinct and no dst may also appear as a src (the host
 * block manager guarantees this: a copy target is a freshly taken block).
 */
PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs,
                         int64_t num_pairs, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, pa_dtype dtype,
                         int *debug_err, void *stream);

/*
 * Bytes of device workspace pa_decode needs for this shape on the current
 * device (depends on its SM count): ~2.5 MB of partial results at head_dim
 * 128 on 152 SMs plus 4 bytes per (sequence, query head).  Returns 0 for
 * invalid arguments.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim);

/*
 * a4 + a5 -- paged decode attention, one query token per sequence:
 *     out[s][h][:] = sum_t softmax_t(scale * <q[s][h], K_t>) V_t
 * over the sequence's whole cached history t = 0 .. context_lens[s]-1, with
 * K_t, V_t read from physical block block_tables[s][t / B], offset t % B, of
 * kv head h / (num_heads / num_kv_heads).  Every new token attends to the
 * whole history (aiqz.cc, section "显存痛点"); the kernel looks the table up
 * before reading each block (cf-1.com news/5879632, section 5.1).  The
 * formula and the grouped-query head mapping are the textbook definition.
 * Arithmetic is fp32 on the stored inputs; out is rounded to nearest even.
 * A sequence with context_len 0 gets a zero row.
 *
 * One kernel launch.  The step's (sequence, kv head, block) tiles are split
 * evenly over one wave of CTAs (split-context); a (sequence, kv head) whose
 * tiles fall in one CTA is finished there, and one cut by range boundaries is
 * combined by the last of its CTAs to finish:
 *     M = max_p m_p;  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
 *
 * workspace: device buffer of at least pa_decode_workspace_size(...) bytes,
 * 16-byte aligned, ZERO-FILLED before its first use.  It holds partial
 * results and per-pair counters; every call leaves the counters at zero
 * again, so a workspace can be reused by later calls of any shape (except
 * after a call that reported PA_DEVERR_TIMEOUT: zero it again then).  Calls
 * that run at the same time need separate workspaces.
 */
PA_API pa_status pa_decode(void *out, const void *q, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables,
                    int max_blocks_per_seq, const int32_t *context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int64_t num_blocks, float scale,
                    pa_dtype dtype, void *workspace, size_t workspace_bytes,
                    int *debug_err, void *stream);

/*
 * a1 + a2 + a4 + a5 in one call: the decode step's K/V write and its decode
 * attention.  Each sequence s with context_lens[s] >= 1 appends one token at
 * position t = context_lens[s] - 1 (the token the step decodes; every new
 * token attends to the whole history including itself, aiqz.cc, section
 * "显存痛点"), so the result is exactly that of
 *     pa_write_kv(new_key[s], new_value[s]) into slot
 *         block_tables[s][t / B] * B + t % B          (for every s), then
 *     pa_decode(...)                                  (same arguments).
 * new_key, new_value: device [num_seqs][num_kv_heads][head_dim], dtype of
 * the pools, 16-byte aligned.  k_cache / v_cache are written (the new rows
 * only).  Sequences with context_len 0 write nothing.  Block ids and
 * positions are range-checked as in pa_slot_mapping (PA_DEVERR bits).
 *
 * Two launches: one kernel looks up every slot and writes the rows (16-byte
 * chunks), then the decode.  On the tensor-core path (fp16 / bf16 pools,
 * block_size % 16 == 0) the decode is launched as a programmatic dependent
 * of the write: it starts while the write runs, sets up its schedule and
 * barriers, and waits for the write to finish before its first read of the
 * pools.  Workspace rules as for pa_decode.
 */
PA_API pa_status pa_write_decode(void *out, const void *q, const void *new_key,
                                 const void *new_value, void *k_cache, void *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int num_seqs, int num_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int64_t num_blocks, float scale, pa_dtype dtype,
                                 void *workspace, size_t workspace_bytes, int *debug_err,
                                 void *stream);

/* Number of CTAs the decode kernel launches on the current device. */
PA_API int pa_decode_grid_size(void);

/*
 * pa_decode for callers that cannot allocate device memory.  The paper has no
 * counterpart to this call; it exists for the library's users.
 *
 * Same arguments and result as pa_decode, without the workspace: the scratch
 * lives in a static 4 MiB device array inside this library (every GPU that
 * loads the library keeps it until the process exits).  Meant for callers
 * that have no device allocator of their own, that must not call cudaMalloc
 * on their path (it can synchronise the whole device), or that run where all
 * device memory is already reserved by someone else.
 *   - Returns PA_ERR_WORKSPACE, and enqueues nothing, when the shape needs more
 *     scratch than 4 MiB (pa_decode_workspace_size(...) > 4 MiB; on a 152-SM
 *     GPU with head_dim 128, when num_seqs * num_heads exceeds about 400 000).
 *   - Allocates nothing.  The first call on a device looks up the array's
 *     device address (cudaGetSymbolAddress), which may load the library's
 *     device code there; make that first call before any stream capture.
 *   - All calls on a device share the one array: calls whose kernels may run
 *     at the same time (unordered streams) race on it.  The array starts
 *     zeroed and every call leaves its counters at zero, so it needs no
 *     clearing between calls (see pa_decode about PA_DEVERR_TIMEOUT).
 */
PA_API pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks,
                                   float scale, pa_dtype dtype, int *debug_err,
                                   void *stream);

/*
 * Plan of a shared-block decode (host, no GPU work).  Sequences that hold the
 * same physical blocks for a common history -- forks of one prompt, whose
 * shared blocks the prefix-sharing passages keep read-only under reference
 * counts (aiqz.cc, section "前缀共享机制"; cf-1.com news/5879632, section
 * 4.1) -- are found from the block tables: groups of two or more sequences
 * whose tables agree on a run of blocks that are full for every member.  The
 * pages read a shared block once per sharer; pa_decode_shared reads it once
 * per group.  Each sequence's blocks past its shared runs (its private blocks,
 * the last one possibly partly filled) form a one-member own group, read by
 * the same kernel.  The plan also splits the groups' work evenly over `nctas` CTAs
 * (pass pa_decode_grid_size()).
 *
 * block_tables, context_lens: HOST int32 arrays [num_seqs][max_blocks_per_seq]
 * and [num_seqs], the same contents the decode will see.  plan: host int32
 * buffer of plan_capacity ints, or NULL to only compute the size.  On return
 * *plan_ints holds the plan's size in ints; PA_ERR_WORKSPACE if plan_capacity
 * is smaller.  The plan stays valid while the tables and lengths keep those
 * contents (or change only in private blocks of the same count) and for the
 * same head counts and nctas.
 */
PA_API pa_status pa_share_plan(const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int block_size,
                               int num_heads, int num_kv_heads, int nctas, int32_t *plan,
                               size_t plan_capacity, size_t *plan_ints);

/*
 * Bytes of device workspace pa_decode_shared needs with this plan (host copy)
 * on the current device; 0 for invalid arguments.
 */
PA_API size_t pa_decode_shared_workspace_size(const int32_t *plan_host, int num_seqs,
                                              int num_heads, int num_kv_heads, int head_dim);

/*
 * pa_decode with each shared block read once per group of sharers.  Same
 * arguments and the same result (up to fp32 rounding order) as pa_decode,
 * plus the plan that pa_share_plan built from these tables: plan_host (host
 * copy, read for its sizes) and plan_dev (device copy of the same ints,
 * 16-byte aligned).  fp16 / bf16 caches with block_size a multiple of 16
 * only (else PA_ERR_UNSUPPORTED).  Up to three launches on `stream`:
 *   1a. the shared groups with 32 or more query rows per kv head (block size
 *      16, 32 or 64), on the tensor cores: one CTA per work item of the plan,
 *      128 query rows against a chunk of the group's run (the plan holds each
 *      item's q rows and physical blocks);
 *   1b. every other group's blocks against the query rows of all its members
 *      (a group is a shared run of full blocks, or one sequence's own blocks),
 *      launched to start while 1a runs: the four consumer warps of a CTA
 *      share each tile, 8 query rows each;
 *      each piece of 1a and 1b leaves a partial state (acc, m, l) per row;
 *   2. per (sequence, head), the merge of the partial states of every group
 *      it belongs to:
 *      M = max_i m_i;  out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
 * workspace: at least pa_decode_shared_workspace_size(...) bytes, 16-byte
 * aligned (the partial states; zero-filled before first use when the plan has
 * no shared group, as pa_decode then runs with it).  A plan without shared
 * groups runs pa_decode.
 */
PA_API pa_status pa_decode_shared(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *context_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, int64_t num_blocks, float scale,
                                  pa_dtype dtype, const int32_t *plan_host,
                                  const int32_t *plan_dev, void *workspace,
                                  size_t workspace_bytes, int *debug_err, void *stream);

/*
 * Prompt (prefill) attention through the block table.  Sequence s owns the
 * query rows q_start[s] .. q_start[s+1]-1 of q / out ([T][num_heads][head_dim],
 * T = q_start[num_seqs]); they are the last n = q_start[s+1] - q_start[s]
 * positions of its context, whose length context_lens[s] counts them, and
 * their K/V are already in the cache (pa_write_kv).  The row at position p
 * attends over tokens 0 .. p: the whole cached history, then the prompt up
 * to itself.  The prompt's tokens enter blocks as the request arrives
 * (cf-1.com news/5879632, section 3.2) and each attends to all history
 * before it (aiqz.cc, section "显存痛点"); the causal mask is the textbook
 * definition.  fp16 / bf16 with block_size 16, 32 or 64 only (else
 * PA_ERR_UNSUPPORTED); head_dim 64 or 128.
 *   q_start     device int32 [num_seqs + 1], q_start[0] = 0, non-decreasing;
 *               a sequence with n > context_lens[s] sets PA_DEVERR_CONTEXT
 *               and is skipped.
 *   max_q_len   host bound of n over the sequences (sizes the grid).
 * One launch on `stream`: one CTA per (sequence, kv head, 128 query rows),
 * tcgen05 MMAs with fp32 accumulators in tensor memory; the probabilities
 * enter the P.V product as two fp16 / bf16 terms (hi + lo), so the result
 * carries fp32-level error; out rounded to nearest even.
 * Allocates nothing; no workspace.
 */
PA_API pa_status pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *q_start, int num_seqs,
                            int max_q_len, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale, pa_dtype dtype,
                            int *debug_err, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
