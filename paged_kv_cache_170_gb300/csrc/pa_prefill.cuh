// pa_prefill.cuh -- prompt (prefill) attention over the paged cache on the
// 5th-generation tensor cores: tcgen05.mma with operands in shared memory
// (TMA-loaded, 128-byte swizzle) or tensor memory, accumulators in tensor
// memory (TMEM).
//
// Sequence s has n new query tokens, the last n positions of its context
// (their K/V already in the cache); the query at position p sees tokens
// 0 .. p.  One CTA takes one (sequence, kv head, tile of 128 query rows); a
// row is (prompt position i, head hh of the kv head's group of G),
// position-major, so all rows share every K/V tile.  The context is consumed
// in steps of 64 tokens (64 / B blocks).  Six warps:
//   warps 0-3  softmax: thread t of warp w owns row 32w + t = TMEM lane
//              32w + t; they stage the Q tile, turn each S into P and write
//              the normalised output.  They also load the keys: each warp
//              its share of a step's K blocks into the K ring as [half][64
//              tokens][128 B] (one 2-D box per block and 64-column half, so a
//              step's keys form one MMA operand), K(j + NKS) into the slot of
//              K(j) once it has seen S_j (QK(j) done);
//   warp 4     producer: streams each step's V blocks into the V ring as
//              [block][half][B tokens][128 B] (one box per block); the lanes
//              hold the block table 32 entries at a time;
//   warp 5     MMA: allocates TMEM and, from one lane, issues every MMA.
// With head_dim 128 the rings hold 2 K and 3 V steps: a K slot is free once
// its QK is done, early in a step, a V slot only once its PV is done.
// Per step j:
//   S_j = Q K_j^T  M = 128 rows, N = the step's tokens, K = D in 16-column
//                  MMAs; A = Q (K-major), B = K (K-major) -> S buffer j % 2;
//   softmax        each thread loads its row of S_j, masks tokens past its
//                  position (only on steps that reach the diagonal or end
//                  short), and forms p = 2^(s * scale * log2 e - m) against a
//                  running maximum m that only moves when the row maximum
//                  exceeds it by more than 8 (l and the row of O are then
//                  rescaled), so most steps never touch O; p goes back into
//                  the same TMEM columns as two 16-bit terms p_hi + p_lo;
//   O += P_j V_j   M = 128, N = D, K = 16 tokens per MMA; A = P from TMEM,
//                  B = V read MN-major (rows = tokens) -> O in TMEM.
// The MMA lane issues PV(i) as soon as P_i and V_i are in and QK(j) as soon
// as K_j is in and PV(j - 2) has been issued (QK(j) overwrites the buffer
// P_{j-2} is read from; MMAs of one thread run in issue order), so the
// softmax of one step overlaps the tensor pipe's work on its neighbours.
// The softmax waits for the previous PV only before it rescales O.  Every
// mbarrier phase is waited by its consumer before the phase after it can
// start (that phase's producer depends on the consumer's next signal), so
// the parity waits are exact; barriers whose consumers may lag are kept per
// step parity.  Rows of a partly filled last block past the context are
// zeroed in the V ring before the PV MMAs read them.  All waits are bounded;
// TMEM is released on every path.
//
// The same kernel also serves the shared-block decode (kGroups): a shared
// group with many sharers is the same contraction -- the query rows of all
// its members (row = member * G + head) against the group's run of shared
// blocks, which every row sees in full.  There a CTA takes one work item of
// the plan (128 rows of one (group, kv head) against a chunk of the run), no
// step is masked but a short last one, and each row leaves its partial state
// (O unnormalised, m, l) in the record of its pass's piece for the merge.
#pragma once

#include "pa_sched.cuh"
#include "pa_share_plan.h"

namespace pagedkv {

struct PrefillArgs {
  void *out;
  const void *q;
  const int32_t *tables;
  const int32_t *lens;
  const int32_t *q_start;  // [S + 1] query rows of each sequence in q / out
  int64_t num_blocks;
  int max_blocks, S, Hq, Hkv, B;
  float qscale;          // scale * log2(e)
  int *err;
  // the shared-block decode's groups (kGroups)
  float *records;        // [piece][kSharePassRows][state_row(D)] partial states
  const int32_t *plan;   // device copy of the plan
  int32_t t_items;       // offset of its TcItem array
  int32_t t_qrow;        // offset of each item's q rows [item][kTcRows]
  int32_t t_blk;         // offset of each item's physical blocks [item][t_blk_stride]
  int32_t t_blk_stride;
};

constexpr int kTcRows = 128;                 // query rows per CTA (= TMEM lanes)
constexpr int kTcStepTokens = 64;            // tokens per softmax step
constexpr int kTcThreads = 6 * 32;
constexpr int kTcMaxSlots = 4;               // step slots per ring, at most
// Step slots of the K and V rings: a K slot is free again once its QK is
// done, early in a step; a V slot only once its PV is done, so V gets one more.
// With head_dim 128: Q 32 KB + K 2 x 16 KB + V 3 x 16 KB = 112 KB, two CTAs per SM.
// The shared-block decode's items (groups) are a few steps long and start
// with a chain of dependent loads: their keys are requested three steps ahead
// (K 3 x 16 KB + V 2 x 16 KB, the same 112 KB).
__host__ __device__ constexpr int tc_k_slots(int D, bool groups = false) { return D == 128 ? (groups ? 3 : 2) : 4; }
__host__ __device__ constexpr int tc_v_slots(int D, bool groups = false) { return D == 128 ? (groups ? 2 : 3) : 4; }
__host__ __device__ constexpr int tc_smem_bytes(int D) {
  return (D / 64) * kTcRows * 128 + (tc_k_slots(D) + tc_v_slots(D)) * (D / 64) * kTcStepTokens * 128;
}
static_assert(tc_k_slots(128, true) + tc_v_slots(128, true) == tc_k_slots(128) + tc_v_slots(128), "same footprint");
constexpr int kTcCols = 256;                 // TMEM columns: O (D) | S/P buffer 0 (64) | S/P buffer 1 (64)

// Shared memory matrix descriptor (tcgen05): 128-byte swizzle, version 1.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A / B of type T,
// A K-major, B K-major (b_mn = false) or MN-major (b_mn = true), M x N.
template <typename T>
__device__ __forceinline__ uint32_t umma_idesc(int M, int N, bool b_mn) {
  const uint32_t ab = Mma<T>::kIsBf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn ? 1u : 0u) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}"
               ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
               : "memory");
}

__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;}"
               ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
               : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane; tmem_ld32_async
// leaves the wait to tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r0)[32], uint32_t (&r1)[32]) {
  // every destination register of both loads is an operand, so no use of one
  // can be scheduled before the wait
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r0[0]), "+r"(r0[1]), "+r"(r0[2]), "+r"(r0[3]), "+r"(r0[4]), "+r"(r0[5]), "+r"(r0[6]), "+r"(r0[7]),
        "+r"(r0[8]), "+r"(r0[9]), "+r"(r0[10]), "+r"(r0[11]), "+r"(r0[12]), "+r"(r0[13]), "+r"(r0[14]), "+r"(r0[15]),
        "+r"(r0[16]), "+r"(r0[17]), "+r"(r0[18]), "+r"(r0[19]), "+r"(r0[20]), "+r"(r0[21]), "+r"(r0[22]), "+r"(r0[23]),
        "+r"(r0[24]), "+r"(r0[25]), "+r"(r0[26]), "+r"(r0[27]), "+r"(r0[28]), "+r"(r0[29]), "+r"(r0[30]), "+r"(r0[31]),
        "+r"(r1[0]), "+r"(r1[1]), "+r"(r1[2]), "+r"(r1[3]), "+r"(r1[4]), "+r"(r1[5]), "+r"(r1[6]), "+r"(r1[7]),
        "+r"(r1[8]), "+r"(r1[9]), "+r"(r1[10]), "+r"(r1[11]), "+r"(r1[12]), "+r"(r1[13]), "+r"(r1[14]), "+r"(r1[15]),
        "+r"(r1[16]), "+r"(r1[17]), "+r"(r1[18]), "+r"(r1[19]), "+r"(r1[20]), "+r"(r1[21]), "+r"(r1[22]), "+r"(r1[23]),
        "+r"(r1[24]), "+r"(r1[25]), "+r"(r1[26]), "+r"(r1[27]), "+r"(r1[28]), "+r"(r1[29]), "+r"(r1[30]), "+r"(r1[31])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// p = p_hi + p_lo in two 16-bit terms per value, packed in pairs.  bf16: p_hi
// is p with its low 16 bits cleared (exact), p_lo = p - p_hi rounded, so the
// pair carries p to about 2^-16 relative.  fp16: p_hi rounded, then the rest.
template <typename T>
struct PSplit {
  static __device__ __forceinline__ void run(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    hi = Mma<T>::pack(p0, p1);
    const float2 f = Mma<T>::unpack(hi);
    lo = Mma<T>::pack(p0 - f.x, p1 - f.y);
  }
};
template <>
struct PSplit<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    const uint32_t b0 = __float_as_uint(p0) & 0xFFFF0000u, b1 = __float_as_uint(p1) & 0xFFFF0000u;
    hi = __byte_perm(b0, b1, 0x7632);
    lo = Mma<__nv_bfloat16>::pack(p0 - __uint_as_float(b0), p1 - __uint_as_float(b1));
  }
};

// One row's step of the online softmax.  Scores s0 (columns 0..31) and s1
// (32..63); with kMask only columns 0 .. nv - 1 are visible.  Moves the
// running maximum m (scaled, base 2) only when the step's maximum exceeds it
// by more than 8; returns the sum of the new p and sets alpha (the factor
// for the old l and O) and the packed p_hi / p_lo.
template <typename T, bool kMask>
__device__ __forceinline__ float softmax_step(const uint32_t (&s0)[32], const uint32_t (&s1)[32], int nv,
                                              float qscale, float &m, float &alpha, uint32_t (&ph)[32],
                                              uint32_t (&pl)[32]) {
  float b0 = -CUDART_INF_F, b1 = -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float x0 = __uint_as_float(s0[c]), x1 = __uint_as_float(s0[c + 1]);
    float y0 = __uint_as_float(s1[c]), y1 = __uint_as_float(s1[c + 1]);
    if (kMask) {
      x0 = c < nv ? x0 : -CUDART_INF_F;
      x1 = c + 1 < nv ? x1 : -CUDART_INF_F;
      y0 = c + 32 < nv ? y0 : -CUDART_INF_F;
      y1 = c + 33 < nv ? y1 : -CUDART_INF_F;
    }
    b0 = fmax3(b0, x0, x1);
    b1 = fmax3(b1, y0, y1);
  }
  const float best = fmaxf(b0, b1);
  const float cand = best == -CUDART_INF_F ? -CUDART_INF_F : best * qscale;
  const bool grow = cand > m + 8.f || (m == -CUDART_INF_F && cand > -CUDART_INF_F);
  const float mnew = grow ? cand : m;
  alpha = (grow && m > -CUDART_INF_F) ? fast_exp2(m - mnew) : 1.f;
  m = mnew;
  const float neg_m = mnew == -CUDART_INF_F ? -CUDART_INF_F : -mnew;
  float lsum0 = 0.f, lsum1 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    // the pair (2c, 2c + 1) of the step's columns
    const int c0 = 2 * c, c1 = 2 * c + 1;
    const float x0 = __uint_as_float(c0 < 32 ? s0[c0 & 31] : s1[c0 & 31]);
    const float x1 = __uint_as_float(c1 < 32 ? s0[c1 & 31] : s1[c1 & 31]);
    float p0 = fast_exp2(fmaf(x0, qscale, neg_m));
    float p1 = fast_exp2(fmaf(x1, qscale, neg_m));
    if (kMask) {
      p0 = c0 < nv ? p0 : 0.f;
      p1 = c1 < nv ? p1 : 0.f;
    }
    lsum0 += p0;
    lsum1 += p1;
    PSplit<T>::run(p0, p1, ph[c], pl[c]);
  }
  return lsum0 + lsum1;
}

// Per-step SM clock stamps of every 256th CTA, and each CTA's SM, start, end
// and step count (PA_TRACE builds only; read back by pa_debug_prefill_trace).
#ifdef PA_TRACE
__device__ long long pa_prefill_steps_trace[16][64][16];
__device__ unsigned long long pa_prefill_cta_trace[16384][3];
#define TC_TRACE(j, f)                                                                          \
  do {                                                                                          \
    if ((blockIdx.x & 255u) == 0 && blockIdx.x < 4096u && (j) < 64)                             \
      pa_prefill_steps_trace[blockIdx.x >> 8][(j)][(f)] = clock64();                            \
  } while (0)
#else
#define TC_TRACE(j, f) \
  do {                 \
  } while (0)
#endif

template <typename T, int D, bool kGroups>
__global__ void __launch_bounds__(kTcThreads, 2)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v) {
  constexpr int HALVES = D / 64;
  constexpr uint32_t QHALF = kTcRows * 128;        // one 64-column half of the Q tile
  constexpr uint32_t SHALF = kTcStepTokens * 128;  // one 64-column half of a step slot
  static_assert(D + 2 * kTcStepTokens <= kTcCols, "TMEM budget");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr uint32_t SS = HALVES * SHALF;  // bytes per step slot
  constexpr int NKS = tc_k_slots(D, kGroups), NVS = tc_v_slots(D, kGroups);
  static_assert(NKS <= kTcMaxSlots && NVS <= kTcMaxSlots, "slots");
  __shared__ __align__(8) uint64_t k_full[kTcMaxSlots];
  __shared__ __align__(8) uint64_t v_full[kTcMaxSlots], v_empty[kTcMaxSlots];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], o_done[2], mma_done;  // [2]: by step parity
  __shared__ uint32_t tmem_base;
  __shared__ int sh_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#ifdef PA_TRACE
  unsigned long long tc_g0, tc_gq = 0, tc_ge = 0, tc_gs[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tc_g0));
#endif
  // the shared-block decode's other step may start launching now: it reads
  // nothing this kernel writes, and fills the SMs this one leaves idle
  if constexpr (kGroups) launch_dependents();
  const int G = a.Hq / a.Hkv;
  const int B = a.B;
  // the CTA's rows r0 .. r0 + 127 (of `rows`), its blocks (ntile physical
  // block ids from trow0 on: the sequence's table row, or for a group the
  // item's block list in the plan), the tokens they hold (L) and, for a
  // prompt, the position of its first query row (pos0) and where its q rows
  // start (q0)
  int kvh, rows, r0, ntile, L, pos0 = 0, q0 = 0;
  const int32_t *trow0;
  int piece[4] = {-1, -1, -1, -1};  // kGroups: the record piece of each pass (32 rows)
  // the Q tile's loads: thread t takes 16-byte chunks t + 128 k (k < kPer), a
  // warp RW rows per k, RK rows apart
  constexpr int kPer = kTcRows * D / 8 / 128, CPR = D / 8, RW = 32 / CPR, RK = kTcRows / CPR;
  const int bps = kTcStepTokens / B;         // blocks per step
  const int kbpw = (bps * HALVES + 3) >> 2;  // K boxes per softmax warp in a full step: 1 or 2
  const int kfirst = (warp & 3) * kbpw;      // this warp's first box
  int kpid0[NKS];                            // lane 0 of a softmax warp: its blocks of the first NKS steps
  int myq = -1;  // kGroups: q row (sequence * Hq + head) of one of this warp's Q rows, -1 past the group's
  if constexpr (kGroups) {
    // the item's q rows and blocks are at fixed strides: requested together
    // with the item itself, one round trip before the Q tile and first keys
    trow0 = a.plan + a.t_blk + (long long)blockIdx.x * a.t_blk_stride;
    if (warp < 4) {
      myq = a.plan[a.t_qrow + (long long)blockIdx.x * kTcRows + RW * warp + lane % RW + RK * (lane / RW)];
      if (lane == 0) {
#pragma unroll
        for (int jj = 0; jj < NKS; ++jj) {
          const int b = jj * bps + kfirst / HALVES;
          kpid0[jj] = b < a.t_blk_stride ? trow0[b] : -1;
        }
      }
    }
    const int4 *it = reinterpret_cast<const int4 *>(a.plan + a.t_items + (long long)blockIdx.x * kTcItemInts);
    const int4 w0 = it[0], w1 = it[1], w2 = it[2];
    kvh = w0.y;
    r0 = w0.z;
    rows = w0.w;
    ntile = w1.w;
    piece[0] = w2.x;
    piece[1] = w2.y;
    piece[2] = w2.z;
    piece[3] = w2.w;
    L = ntile * B;  // shared blocks are full
    if (ntile <= 0 || ntile > a.t_blk_stride || r0 >= rows) {
      if (threadIdx.x == 0) raise_error(a.err, PA_DEVERR_CONTEXT);  // not an item the planner makes
      return;
    }
  } else {
    // heaviest tiles first over all (sequence, kv head) pairs
    const int pairs = a.S * a.Hkv;
    const int pair = int(blockIdx.x % unsigned(pairs));
    const int qt = int(gridDim.x / unsigned(pairs)) - 1 - int(blockIdx.x / unsigned(pairs));
    const int s = pair / a.Hkv;
    kvh = pair % a.Hkv;
    q0 = a.q_start[s];
    const int n = a.q_start[s + 1] - q0;
    const long long cap = (long long)a.max_blocks * B;
    long long Lr = a.lens[s];
    Lr = Lr < 0 ? 0 : (Lr > cap ? cap : Lr);
    L = int(Lr);
    if (n < 0 || n > L) {
      if (threadIdx.x == 0 && qt == 0 && kvh == 0) raise_error(a.err, PA_DEVERR_CONTEXT);
      return;
    }
    rows = n * G;
    r0 = qt * kTcRows;
    if (r0 >= rows) return;
    pos0 = L - n;
    const int p_last = pos0 + (min(rows, r0 + kTcRows) - 1) / G;
    ntile = p_last / B + 1;
    trow0 = a.tables + (long long)s * a.max_blocks;
  }
  const int nstep = (ntile + bps - 1) / bps;

  // shared memory: Q tile, K ring, V ring.  The swizzled tiles need a
  // 1024-byte aligned base; the launch reserves no slack for it (two CTAs
  // fill an SM exactly), so a misaligned base is reported and nothing done.
  const uint32_t raw = smem_addr(smem_raw);
  if (raw & 1023u) {
    if (threadIdx.x == 0) raise_error(a.err, PA_DEVERR_LAYOUT);
    return;
  }
  unsigned char *qs = smem_raw;
  unsigned char *kring = qs + HALVES * QHALF;
  unsigned char *vring = kring + size_t(NKS) * SS;
  const uint32_t q_addr = raw;
  const uint32_t kring_addr = q_addr + HALVES * QHALF, vring_addr = kring_addr + uint32_t(NKS) * SS;
  volatile int *abort_flag = &sh_abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcMaxSlots; ++i) {
      mbar_init(&k_full[i], 4);  // one arrival per softmax warp (each loads its share of a step's keys)
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], 4);
    mbar_init(&p_full[1], 4);
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    mbar_init(&mma_done, 1);
    sh_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();  // the barriers are initialised; the producer starts at once
  if (threadIdx.x == 0) TC_TRACE(0, 11);

  // Keys: each softmax warp loads its share of every step's K boxes (one 2-D
  // box per block and 64-column half, into the step's K slot as [half][64
  // tokens][128 B]); a warp's boxes lie in one block.  K(j + NKS) goes into
  // the slot of K(j) as soon as the warp sees S_j, i.e. QK(j) done.
  const int32_t *ktrow = trow0;
  auto k_entry = [&](int jj) {                   // the table entry of this warp's block of step jj
    const int b = jj * bps + kfirst / HALVES;
    return (jj < nstep && b < ntile) ? ktrow[b] : 0;
  };
  auto k_issue = [&](int jj, int pid) {          // lane 0
    const int nb = min(bps, ntile - jj * bps);
    const int cnt = max(0, min(kbpw, nb * HALVES - kfirst));
    const bool in_pool = pid >= 0 && pid < a.num_blocks;
    if (cnt > 0 && !in_pool) raise_error(a.err, PA_DEVERR_BLOCK_ID);  // block 0 is loaded in its place
    const int y = ((in_pool ? pid : 0) * a.Hkv + kvh) * B;
    uint64_t *bar = &k_full[jj % NKS];
    mbar_arrive_expect_tx(bar, uint32_t(cnt) * uint32_t(B) * 128u);
    for (int e = 0; e < cnt; ++e) {
      const int box = kfirst + e, blk = box / HALVES, hh = box % HALVES;
      tma_load_2d(kring + size_t(jj % NKS) * SS + hh * SHALF + blk * B * 128, &map_k, 64 * hh, y, bar);
    }
  };
  int kpid_next = 0;  // lane 0 of a softmax warp: the entry of K(j + NKS) while step j runs
  int kissued = 0;    // steps whose keys this warp has requested

  if (warp < 4) {
    // ---- the Q tile: rows r0 .. r0 + 127, K-major halves [128 rows][128 B],
    // swizzled; every load is issued before the first store
    const int t = threadIdx.x;  // 0..127
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
      if constexpr (!kGroups) {
#pragma unroll
        for (int jj = 0; jj < NKS; ++jj) kpid0[jj] = k_entry(jj);
      }
      kpid_next = k_entry(NKS);
    }
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = t + 128 * k;
      const int r = i / CPR, c = i % CPR;  // row, 16-byte chunk
      const int gr = r0 + r;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (kGroups) {
        const int qi = __shfl_sync(kFullMask, myq, lane / CPR + RW * k);  // row r's q row
        if (qi >= 0) v[k] = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.q) + (long long)qi * D + c * 8);
      } else if (gr < rows) {
        v[k] = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.q) +
                                                ((long long)(q0 + gr / G) * a.Hq + kvh * G + gr % G) * D + c * 8);
      }
    }
    if (lane == 0) {  // the first NKS steps' keys, while the Q loads are in flight
#pragma unroll
      for (int jj = 0; jj < NKS; ++jj)
        if (jj < nstep) k_issue(jj, kpid0[jj]);
      kissued = min(NKS, nstep);
    }
    const uint32_t flip = a.qscale < 0.f ? 0x80008000u : 0u;  // S of -q with |scale|: the softmax only looks for maxima
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = t + 128 * k;
      const int r = i / (D / 8), c = i % (D / 8);
      const uint4 w = make_uint4(v[k].x ^ flip, v[k].y ^ flip, v[k].z ^ flip, v[k].w ^ flip);
      *reinterpret_cast<uint4 *>(qs + (c >> 3) * QHALF + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = w;
    }
    fence_proxy_async_shared();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "n"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the softmax and MMA warps meet once the Q tile is staged and TMEM allocated
  if (warp != 4) {
    tc_fence_before();
    named_barrier_sync(1, 5 * 32);
    tc_fence_after();
  }
  const uint32_t tmem = warp != 4 ? tmem_base : 0u;  // the producer never touches TMEM
#ifdef PA_TRACE
  if (threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tc_gq));
#endif

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; lane 0 polls the barriers and issues the
    // copies of the values.  The lanes hold the table entries of the current
    // 32 blocks, the next 32 already requested.
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_v)) : "memory");
    const int32_t *trow = trow0;
    const uint32_t tile_bytes = uint32_t(B) * D * 2;
    auto entry = [&](int b) { return b < ntile ? trow[b] : -1; };
    int cur = entry(lane), nxt = entry(32 + lane), chunk = 0;
    // A step's V blocks go to a V slot as [block][half][B tokens][128 B]
    // (one box per block).  A step's blocks lie in one 32-block chunk (the
    // blocks per step divide 32).  A table entry outside the pool raises the
    // error and loads block 0 in its place, so the byte count is always nb
    // tiles.
    auto load_step = [&](unsigned char *dst, uint64_t *bar, int j) {
      const int b0 = j * bps, nb = min(bps, ntile - b0);
      if (b0 >> 5 != chunk) {
        cur = nxt;
        chunk = b0 >> 5;
        nxt = entry(((chunk + 1) << 5) + lane);
      }
      int y[4];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pid = __shfl_sync(kFullMask, cur, (b0 + i) & 31);
        const bool in_pool = pid >= 0 && pid < a.num_blocks;
        bad = bad || (i < nb && !in_pool);
        y[i] = ((in_pool ? pid : 0) * a.Hkv + kvh) * B;
      }
      if (lane == 0) {
        if (bad) raise_error(a.err, PA_DEVERR_BLOCK_ID);
        mbar_arrive_expect_tx(bar, uint32_t(nb) * tile_bytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i >= nb) break;
          if (HALVES == 2)
            tma_load_3d(dst + i * 2 * B * 128, &map_v, 0, y[i], 0, bar);
          else
            tma_load_2d(dst + i * B * 128, &map_v, 0, y[i], bar);
        }
      }
    };
    int vj = 0;
    long long t_last = clock64();
    while (vj < nstep) {
      const int slot = vj % NVS;
      const uint32_t use = uint32_t(vj / NVS);
      const bool free_slot =
          __shfl_sync(kFullMask, use == 0 || (lane == 0 && mbar_test_wait(&v_empty[slot], (use - 1) & 1u)), 0);
      if (free_slot) {
        if (lane == 0) TC_TRACE(vj, 13);
        load_step(vring + size_t(slot) * SS, &v_full[slot], vj);
        if (lane == 0) TC_TRACE(vj, 10);
        ++vj;
        t_last = clock64();
        continue;
      }
      __nanosleep(32);  // nothing to issue: leave the issue slots to the softmax warps for a moment
      const bool stop = __shfl_sync(kFullMask, *abort_flag != 0 || clock64() - t_last > kWaitLimitCycles, 0);
      if (stop) {
        if (lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          raise_error(a.err, PA_DEVERR_TIMEOUT);
        }
        break;
      }
    }
    // no copy into this CTA's shared memory may still be in flight at the end
    if (lane == 0) {
      int never = 0;
      for (int slot = 0; slot < NVS; ++slot)
        if (vj > slot) mbar_wait(&v_full[slot], uint32_t((vj - 1 - slot) / NVS) & 1u, &never);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t id_pv = umma_idesc<T>(kTcRows, D, true);
      // descriptors are built once; the address field counts 16-byte units,
      // so an offset inside shared memory is added to it directly
      const uint64_t qd0 = umma_desc_sw128(q_addr, 16, 1024);
      const uint64_t kd0 = umma_desc_sw128(kring_addr, 16, 1024);
      const uint64_t vd0 = umma_desc_sw128(vring_addr, uint32_t(B) * 128, 1024);  // LBO: the halves of a V block
      uint32_t vofs[4];  // the step's 16-token k-steps in a V slot ([block][half][B][128 B])
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int t = kk * 16;
        vofs[kk] = uint32_t((t / B) * HALVES * B * 128 + (t % B) * 128) >> 4;
      }
      // Issue PV(i) once P_i and V_i are in, and QK(j) once K_j is in and
      // PV(j - 2) has been issued (QK(j) overwrites the buffer P_{j-2} is
      // read from; MMAs of one thread run in issue order).
      bool ok = true;
      int nq = 0, np = 0;  // QKs and PVs issued
      long long t_last = clock64();
      while (np < nstep) {
        bool prog = false;
        if (np < nq && mbar_test_wait(&p_full[np & 1], uint32_t(np >> 1) & 1u) &&
            mbar_test_wait(&v_full[np % NVS], uint32_t(np / NVS) & 1u)) {  // O += P_i V_i
          const int i = np;
          const int nkk = min(bps, ntile - i * bps) * B / 16;
          const int slot = i % NVS;
          TC_TRACE(i, 7);
          tc_fence_after();
          const uint64_t vd = vd0 + ((uint32_t(slot) * SS) >> 4);
          const uint32_t pb = tmem + uint32_t(D + kTcStepTokens * (i & 1));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (kk < nkk) {
              umma_ts(tmem, pb + kk * 8, vd + vofs[kk], id_pv, (i > 0 || kk > 0) ? 1u : 0u);
              umma_ts(tmem, pb + 32 + kk * 8, vd + vofs[kk], id_pv, 1u);
            }
          }
          TC_TRACE(i, 15);
          umma_commit(&v_empty[slot]);
          umma_commit(&o_done[i & 1]);
          TC_TRACE(i, 8);
          ++np;
          prog = true;
        }
        if (nq < nstep && nq <= np + 1 && mbar_test_wait(&k_full[nq % NKS], uint32_t(nq / NKS) & 1u)) {
          const int j = nq;  // S_j = Q K_j^T into buffer j % 2
          const int nb = min(bps, ntile - j * bps);
          const int slot = j % NKS;
          TC_TRACE(j, 4);
          tc_fence_after();
          const uint64_t kd = kd0 + ((uint32_t(slot) * SS) >> 4);
          const uint32_t id_qk = umma_idesc<T>(kTcRows, nb * B, false);
          const uint32_t sb = tmem + uint32_t(D + kTcStepTokens * (j & 1));
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            umma_ss(sb, qd0 + uint32_t(((ks >> 2) * QHALF + (ks & 3) * 32) >> 4),
                    kd + uint32_t(((ks >> 2) * SHALF + (ks & 3) * 32) >> 4), id_qk, ks > 0 ? 1u : 0u);
          umma_commit(&s_full[j & 1]);
          TC_TRACE(j, 5);
          ++nq;
          prog = true;
        }
        if (prog) {
          t_last = clock64();
        } else if (*abort_flag || clock64() - t_last > kWaitLimitCycles) {
          ok = false;
          break;
        } else if (np < nq) {
          // nothing ready: suspend on the likeliest next event (the softmax
          // warps' P_i) instead of spinning on the issue slots they share
          mbar_try_wait(&p_full[np & 1], uint32_t(np >> 1) & 1u);
        } else {
          mbar_try_wait(&k_full[nq % NKS], uint32_t(nq / NKS) & 1u);
        }
      }
      if (!ok && !*abort_flag) {
        *abort_flag = 1;
        raise_error(a.err, PA_DEVERR_TIMEOUT);
      }
      // every MMA this thread issued has finished before TMEM is released
      umma_commit(&mma_done);
      int never = 0;
      mbar_wait(&mma_done, 0u, &never);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int row = warp * 32 + lane;  // TMEM lane
    const int gr = r0 + row;
    const int pos = pos0 + gr / G;
    const int pos_first = pos0 + r0 / G;
    const uint32_t tl = tmem + (uint32_t(warp * 32) << 16);
    const float qscale = fabsf(a.qscale);  // Q was negated for a negative scale
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nstep; ++j) {
      const int t0 = j * kTcStepTokens;
      const int nb = min(bps, ntile - j * bps);
      ok = ok && !*abort_flag && mbar_wait(&s_full[j & 1], uint32_t(j >> 1) & 1u, abort_flag);
      ok = __all_sync(kFullMask, ok);
      if (!ok) break;
      if (threadIdx.x == 0) TC_TRACE(j, 0);
#ifdef PA_TRACE
      if (threadIdx.x == 0 && j < 8) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tc_gs[j]));
#endif
      tc_fence_after();
      const uint32_t sb = tl + uint32_t(D + kTcStepTokens * (j & 1));
      // a partly filled last block: zero its V rows past the context before the PV MMAs read them
      if (j == nstep - 1 && L < ntile * B) {
        const int slot = j % NVS;
        ok = mbar_wait(&v_full[slot], uint32_t(j / NVS) & 1u, abort_flag);
        ok = __all_sync(kFullMask, ok);
        if (!ok) break;
        // the last block of the slot ([block][half][B][128 B]); its rows zfrom .. B - 1
        unsigned char *vs = vring + size_t(slot) * SS + size_t(ntile - 1 - j * bps) * HALVES * B * 128;
        const int zfrom = L - (ntile - 1) * B;
        for (int i = threadIdx.x; i < (B - zfrom) * HALVES * 8; i += 128) {
          const int r = zfrom + i / (HALVES * 8);
          const int hc = i % (HALVES * 8);
          *reinterpret_cast<uint4 *>(vs + (hc >> 3) * B * 128 + r * 128 + (hc & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_shared();
      }
      uint32_t s0[32], s1[32];
      tmem_ld32_async(sb, s0);
      tmem_ld32_async(sb + 32, s1);
      tmem_wait_ld(s0, s1);
      // only steps that reach the diagonal or end short need a mask; the
      // visible columns of a row are then a prefix 0 .. nv - 1 (a group's
      // rows see every token: only a short last step is masked)
      const bool need_mask =
          kGroups ? nb * B < kTcStepTokens : (t0 + kTcStepTokens - 1 > pos_first || nb * B < kTcStepTokens);
      uint32_t ph[32], pl[32];
      float alpha, lsum;
      if (need_mask)
        lsum = softmax_step<T, true>(s0, s1, kGroups ? nb * B : min(nb * B, pos - t0 + 1), qscale, m, alpha, ph,
                                     pl);
      else
        lsum = softmax_step<T, false>(s0, s1, kTcStepTokens, qscale, m, alpha, ph, pl);
      l = l * alpha + lsum;
      if (threadIdx.x == 0) TC_TRACE(j, 1);
      // a rescale of O waits for the previous step's PV (PV(j) waits for
      // this warp's P_j); P_j itself goes to the other buffer, so a step
      // that keeps its maximum does not wait for the tensor pipe
      if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
        ok = mbar_wait(&o_done[(j - 1) & 1], uint32_t((j - 1) >> 1) & 1u, abort_flag);
        ok = __all_sync(kFullMask, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tl + c0, ov);
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          tmem_st32(tl + c0, ov);
        }
      }
      if (threadIdx.x == 0) TC_TRACE(j, 2);
      tmem_st32(sb, ph);
      tmem_st32(sb + 32, pl);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
      if (lane == 0) {  // trace: each softmax warp's release of P_j (warp 0: field 3; warps 1-3: 6, 12, 14)
        if (warp == 0) TC_TRACE(j, 3);
        else if (warp == 1) TC_TRACE(j, 6);
        else if (warp == 2) TC_TRACE(j, 12);
        else TC_TRACE(j, 14);
      }
      // QK(j) is done (S_j was read): its K slot takes K(j + NKS); issued
      // once P_j is out, off the path from S_j to P_j
      if (lane == 0 && j + NKS < nstep) {
        k_issue(j + NKS, kpid_next);
        ++kissued;
        kpid_next = k_entry(j + NKS + 1);
        if (warp == 0) TC_TRACE(j + NKS, 9);
      }
    }
    // ---- the output row: O / l
    if (ok) {
      ok = mbar_wait(&o_done[(nstep - 1) & 1], uint32_t((nstep - 1) >> 1) & 1u, abort_flag);
      ok = __all_sync(kFullMask, ok);
    }
#ifdef PA_TRACE
    if (threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tc_ge));
#endif
    if (ok && kGroups) {
      // the row's partial state (O, m, l) in the record of its pass's piece:
      // softmax warp w holds pass 4 * (r0 / 128) + w, row lane of it
      tc_fence_after();
      constexpr int R = state_row(D);
      float *rec = gr < rows ? a.records + ((long long)piece[warp] * kSharePassRows + lane) * R : nullptr;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tmem_ld32(tl + c0, ov);
        if (rec != nullptr) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4 *>(rec + c0 + c) = make_float4(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1]),
                                                                    __uint_as_float(ov[c + 2]), __uint_as_float(ov[c + 3]));
        }
      }
      if (rec != nullptr) {
        rec[D] = m;
        rec[D + 1] = l;
      }
    } else if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      T *orow = static_cast<T *>(a.out) + ((long long)(q0 + gr / G) * a.Hq + kvh * G + gr % G) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tmem_ld32(tl + c0, ov);
        if (gr < rows) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = Mma<T>::pack(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(orow + c0 + 8 * c) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                                                                       pk[4 * c + 3]);
        }
      }
    } else if (lane == 0) {
      *abort_flag = 1;
      raise_error(a.err, PA_DEVERR_TIMEOUT);
    }
    // after an abort no key copy of this warp may still be in flight at the
    // end (on the normal path every one was waited for before its QK)
    if (!ok && lane == 0) {
      int never = 0;
      for (int slot = 0; slot < NKS; ++slot)
        if (kissued > slot) mbar_wait(&k_full[slot], uint32_t((kissued - 1 - slot) / NKS) & 1u, &never);
    }
  }

  // ---- every role is done with TMEM (the MMA lane waited for its last MMA)
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcCols));
  }
#ifdef PA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 16384u) {  // every CTA: start and end (global ns timer), SM, steps
    unsigned long long g1;
    unsigned sm;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g1));
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    pa_prefill_cta_trace[blockIdx.x][0] = tc_g0;
    pa_prefill_cta_trace[blockIdx.x][1] = g1;
    pa_prefill_cta_trace[blockIdx.x][2] = (uint64_t(sm) << 32) | uint32_t(nstep);
    if (kGroups)  // the groups mode's timeline: start, Q staged, S_0 .. S_3 seen, epilogue, end
      printf("tracetc %d %u %llu %llu %llu %llu %llu %llu %llu %llu %d\n", blockIdx.x, sm, tc_g0, tc_gq, tc_gs[0],
             tc_gs[1], tc_gs[2], tc_gs[3], tc_ge, g1, nstep);
  }
#endif
}

}  // namespace pagedkv
