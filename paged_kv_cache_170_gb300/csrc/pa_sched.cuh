// pa_sched.cuh -- work schedule shared by the two decode kernels.
//
// The step's work is the ordered list of tiles (sequence s, pair-chunk pc,
// logical block b), pc = kv head * HC + head chunk, where a head chunk is GT
// of the G query heads that share one kv head and a tile is one physical
// block of K plus the same block of V for that kv head.  The W tiles are cut
// into N contiguous ranges of equal cost, one per CTA (N = one full wave, 2
// CTAs per SM), a tile costing 1 and each (s, pc) segment kSegCost more: every
// CTA streams about the same number of bytes, fewer when its range holds many
// short segments, whatever the length mix.
// A CTA finishes any (s, pc) whose tiles all fall in its range and writes
// `out`; a (s, pc) cut by a range boundary leaves a partial (acc, m, l) for
// the pair's last contributor to merge: slot 0 for the CTA's first segment,
// slot 1 for its last.
#pragma once

#include <math_constants.h>

#include "pa_common.cuh"

#ifdef PA_TRACE
#ifndef PA_TRACE_CTA
#define PA_TRACE_CTA(c) ((c) % 101 == 0)  // CTAs whose warps print their counters
#endif
#endif

namespace pagedkv {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = kConsumerWarps;       // fills the ring
constexpr int kMergerWarp = kConsumerWarps + 1;     // combines the consumers' states
constexpr int kDecodeThreads = (kConsumerWarps + 2) * 32;
constexpr int kCtasPerSm = 2;
constexpr int kMaxStages = 64;
constexpr int kMaxBlockSize = 64;
constexpr int kRingBytes = 80 * 1024;      // CUDA-core kernel: ring of K + V tile pairs
constexpr int kRingBytesMma = 90 * 1024;   // tensor-core kernel: K + V tiles + the segment's q rows
constexpr int kMergeRecords = 32;  // records whose merge weights are staged in shared memory
constexpr int kMergeScratch = 2 * kMergeRecords * 8 + kMergeRecords;  // floats: m, l per (record, head); record ids

struct DecodeArgs {
  void *out;
  const void *q;
  const char *k_cache;
  const char *v_cache;
  const int32_t *tables;
  const int32_t *lens;
  int64_t num_blocks;
  int max_blocks;
  int S, Hq, Hkv, B;
  float qscale;            // scale * log2(e)
  float *partials;         // [N][2][8][state_row(D)]: acc[D], m, l per head
  unsigned *counters;      // [S * PC] contributors seen per split pair; zero between calls
  int *err;
  int nctas;
  int nstage;
  uint32_t slot_stride;    // bytes between ring slots (one slot = K tile + V tile)
  uint32_t tile_stride;    // offset of the V tile inside a slot
  int GT;                  // query heads per pair-chunk (<= 8)
  int ncw;                 // consumer warps that take tiles
  int pg;                  // ring entries the producer issues at once (ncw + pg <= nstage)
  int nops;                // tensor copies per tile (1: one 3-D box; 2: two 2-D halves)
  uint32_t q_offset;       // tensor-core kernel: offset of the q rows inside a slot
  uint32_t q_bytes;        // tensor-core kernel: bytes of q rows of one pair chunk (GT * D * e)
};

// Output row `row` (= s * Hq + hq), dims d .. d+3 (store_out4) or d.
template <typename T>
__device__ __forceinline__ void store_out4(const DecodeArgs &a, long long row, int d, int D, float4 v) {
  Elem<T>::store4(static_cast<T *>(a.out) + row * D + d, v);
}

template <typename T>
__device__ __forceinline__ void store_out1(const DecodeArgs &a, long long row, int d, int D, float v) {
  static_cast<T *>(a.out)[row * D + d] = Elem<T>::from_float(v);
}

// Wait until ring entry e (slot e % nstage, its u-th use, u = e / nstage) has
// landed.  An entry is one tile pair.  Consumer warps take pairs round-robin,
// so the warp waiting for use u of a slot is in general not the one that
// consumed use u - 1, and an mbarrier parity wait is only unambiguous while
// the barrier is at most one phase behind.  So first wait until use u - 1 was
// released (phase u - 1 of the slot's empty barrier): that release implies
// use u - 1 landed.  The release barrier itself is never more than one phase
// behind: a warp reaching pair e has consumed pair e - ncw, so the producer
// finished every group of pg entries before the one holding e - ncw, which
// includes e - nstage when ncw + pg <= nstage, and issuing e - nstage
// required use u - 2 to be released.
__device__ __forceinline__ bool wait_entry(uint64_t *full, uint64_t *empty, uint32_t e, int nstage,
                                           volatile int *abort) {
  const int slot = int(e % uint32_t(nstage));
  const uint32_t u = e / uint32_t(nstage);
  if (u > 0 && !mbar_wait(&empty[slot], (u - 1) & 1u, abort)) return false;
  return mbar_wait(&full[slot], u & 1u, abort);
}

// Context length of sequence s clamped to its table's capacity (the scan
// flags lengths outside [0, max_blocks * B]).
__device__ __forceinline__ int clamped_len(const DecodeArgs &a, int s) {
  int L = a.lens[s];
  const int cap = a.max_blocks * a.B;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// Tokens of sequence s the decode attends over: its clamped length.
__device__ __forceinline__ int eff_len(const DecodeArgs &a, int s) { return clamped_len(a, s); }

__device__ __forceinline__ int blocks_of(const DecodeArgs &a, int s) {
  return (eff_len(a, s) + a.B - 1) / a.B;
}

// The step's tiles are flattened in (s, pc, block) order; a segment is the nb
// tiles of one (s, pc).  CTAs split the step by cost, not by tiles: a segment
// costs kSegCost + nb, so that CTAs whose range holds many short segments
// (their hand-offs and merges, about 2.6k SM cycles each, measured) get fewer
// tiles.  Tile b of a segment whose cost range starts at Cp sits at cost
// position Cp + kSegCost + b; CTA c owns the tiles at positions
// [ceil(c Wc / N), ceil((c + 1) Wc / N)), i.e. the tile at position P
// belongs to CTA floor(P N / Wc).
constexpr int kSegCost = 4;

__device__ __forceinline__ long long seg_cost(int nb) { return nb > 0 ? (long long)nb + kSegCost : 0; }

// Where a key falls: by tile index (by_cost false) or by cost position.  Run
// by one whole warp; the key must be < W (resp. < Wc).  Returns the
// sequence, the tile offset inside it (for a cost position inside a
// segment's fixed cost: that segment's first tile), the tiles and the cost
// before the sequence.
__device__ __forceinline__ void locate(const DecodeArgs &a, int PC, int lane, long long key, bool by_cost,
                                       int *s_out, long long *r_out, long long *texcl_out, long long *cexcl_out) {
  int sx = a.S;
  long long rx = 0, tx = 0, cx = 0, run = 0, crun = 0;
  for (int base = 0; base < a.S && sx == a.S; base += 32) {
    const int s = base + lane;
    const int nb = s < a.S ? blocks_of(a, s) : 0;
    const long long n = (long long)nb * PC, c = seg_cost(nb) * PC;
    long long incl = n, cincl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(kFullMask, incl, off);
      const long long cy = __shfl_up_sync(kFullMask, cincl, off);
      if (lane >= off) {
        incl += y;
        cincl += cy;
      }
    }
    const long long excl = run + incl - n, cexcl = crun + cincl - c;
    const bool hit = by_cost ? (c > 0 && cexcl <= key && key < crun + cincl) : (n > 0 && excl <= key && key < run + incl);
    const unsigned m = __ballot_sync(kFullMask, hit);
    if (m) {
      const int leader = __ffs(m) - 1;
      long long r = key - excl;
      if (by_cost && hit) {
        const long long rc = key - cexcl, sc = seg_cost(nb);
        const long long o = rc % sc - kSegCost;
        r = (rc / sc) * nb + (o > 0 ? o : 0);
      }
      sx = __shfl_sync(kFullMask, s, leader);
      rx = __shfl_sync(kFullMask, r, leader);
      tx = __shfl_sync(kFullMask, excl, leader);
      cx = __shfl_sync(kFullMask, cexcl, leader);
    }
    run += __shfl_sync(kFullMask, incl, 31);
    crun += __shfl_sync(kFullMask, cincl, 31);
  }
  *s_out = sx;
  *r_out = rx;
  *texcl_out = tx;
  *cexcl_out = cx;
}

// The CTA's plan.  W = total tiles of the step, Wc their total cost; the CTA
// owns the tiles [w0, w1).  It processes its range rotated: first [Ls, w1),
// the segment that ends the range (usually the head of a (s, pc) cut by the
// range end), then [w0, Ls).  Both ends of a cut (s, pc) are then worked on
// early by the two CTAs that share it, so their merge overlaps with
// streaming instead of piling up at the end of the kernel.  (sA, rA, cA) /
// (s0, r0, c0) locate Ls / w0: sequence, tile offset inside it, cost position
// where the segment holding that tile starts.
struct Plan {
  long long W, Wc, w0, w1, Ls;
  int sA, s0;
  long long rA, r0, cA, c0;
};

// First tile at cost position >= t.
__device__ __forceinline__ long long tile_at_cost(const DecodeArgs &a, int PC, int lane, long long t, long long W,
                                                  long long Wc) {
  if (t >= Wc) return W;
  int s;
  long long r, te, ce;
  locate(a, PC, lane, t, true, &s, &r, &te, &ce);
  return te + r;
}

// CTA that owns the tile at cost position P, and whether CTA c owns any tile.
__device__ __forceinline__ int cta_at_cost(long long P, long long Wc, int N) { return int(P * N / Wc); }
__device__ __forceinline__ long long cost_start(int c, long long Wc, int N) { return ((long long)c * Wc + N - 1) / N; }

__device__ __forceinline__ void schedule_scan(const DecodeArgs &a, int PC, int lane, Plan *plan) {
  const int cap = a.max_blocks * a.B;
  long long run = 0, crun = 0;
  for (int base = 0; base < a.S; base += 32) {
    const int s = base + lane;
    long long n = 0, c = 0;
    if (s < a.S) {
      const int L = a.lens[s];
      if ((L < 0 || L > cap) && blockIdx.x == 0) raise_error(a.err, PA_DEVERR_CONTEXT);
      const int nb = blocks_of(a, s);
      n = (long long)nb * PC;
      c = seg_cost(nb) * PC;
    }
    long long incl = n, cincl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(kFullMask, incl, off);
      const long long cy = __shfl_up_sync(kFullMask, cincl, off);
      if (lane >= off) {
        incl += y;
        cincl += cy;
      }
    }
    run += __shfl_sync(kFullMask, incl, 31);
    crun += __shfl_sync(kFullMask, cincl, 31);
  }
  Plan p;
  p.W = run;
  p.Wc = crun;
  p.w0 = tile_at_cost(a, PC, lane, cost_start(blockIdx.x, p.Wc, a.nctas), p.W, p.Wc);
  p.w1 = tile_at_cost(a, PC, lane, cost_start(blockIdx.x + 1, p.Wc, a.nctas), p.W, p.Wc);
  p.Ls = p.w0;
  p.sA = p.s0 = a.S;
  p.rA = p.r0 = p.cA = p.c0 = 0;
  if (p.w0 < p.w1) {
    long long te, ce;
    locate(a, PC, lane, p.w0, false, &p.s0, &p.r0, &te, &ce);
    const int nb0 = blocks_of(a, p.s0);
    p.c0 = ce + (p.r0 / nb0) * seg_cost(nb0);
    int sl;
    long long rl;
    locate(a, PC, lane, p.w1 - 1, false, &sl, &rl, &te, &ce);
    const int nb = blocks_of(a, sl);
    const long long pair_start = (p.w1 - 1) - rl % nb;
    if (pair_start > p.w0) {
      p.Ls = pair_start;
      p.sA = sl;
      p.rA = rl - rl % nb;
      p.cA = ce + (rl / nb) * seg_cost(nb);
    } else {
      p.sA = p.s0;
      p.rA = p.r0;
      p.cA = p.c0;
    }
  }
  *plan = p;
}

// Processing order of a CTA's range: phase 0 walks [Ls, w1), phase 1 [w0, Ls).
__device__ __forceinline__ bool phase_range(const Plan &p, int ph, long long *from, long long *to) {
  *from = ph == 0 ? p.Ls : p.w0;
  *to = ph == 0 ? p.w1 : p.Ls;
  return *from < *to;
}

// Cursor over a CTA's tile range, one segment (consecutive tiles of one
// (s, pc)) at a time.  Producer and consumers walk identical sequences.
struct Walk {
  int s, pc, b, nb, L;  // L: tokens of s (eff_len, read once per sequence)
  long long w;
  long long cp;         // cost position where the current segment starts
  __device__ __forceinline__ void start(const DecodeArgs &a, int s0, long long r0, long long w0, long long c0) {
    s = s0;
    L = eff_len(a, s);
    nb = (L + a.B - 1) / a.B;
    pc = int(r0 / nb);
    b = int(r0 % nb);
    w = w0;
    cp = c0;
  }
  __device__ __forceinline__ int seg_len(long long w1) const {
    return int((long long)(nb - b) < w1 - w ? (long long)(nb - b) : w1 - w);
  }
  __device__ __forceinline__ void advance(const DecodeArgs &a, int n, int PC) {
    w += n;
    b += n;
    if (b == nb) {
      b = 0;
      cp += seg_cost(nb);
      if (++pc == PC) {
        pc = 0;
        do {
          ++s;
        } while (s < a.S && blocks_of(a, s) == 0);
        if (s < a.S) {
          L = eff_len(a, s);
          nb = (L + a.B - 1) / a.B;
        }
      }
    }
  }
};

// The producer warp: walks the CTA's range, reads the block table 32 entries
// at a time (coalesced, next batch prefetched, kept in registers: never
// re-read per token) and fills the ring.  Entries are issued in groups of pg:
// lane i < pg claims entry e + i (waits until its slot's previous use was
// released) and calls issue(slot, pid, kv head, logical block, context len,
// s, pc, lead), which announces the bytes on full_bar[slot] and starts the
// copies; the lanes of a group wait and issue in parallel.  `lead` marks the
// first ncw entries of a segment: every consumer warp that takes part in the
// segment meets one of them first, so a kernel can ship per-segment data
// (the q rows) with those entries only.  issued[slot] keeps the last use
// issued into each slot so the producer can wait for every copy still in
// flight before it leaves (after an abort too).
//
// The producer's copies are the kernel's first reads of the pools, so it is
// where the kernel waits for the grid it depends on (griddepcontrol.wait: a
// no-op unless the launch allowed an early start, as pa_write_decode's does,
// so that the plan and the barriers are set up while the previous kernel
// runs).
template <class Issue>
__device__ __forceinline__ void produce(const DecodeArgs &a, int PC, int HC, const Plan &plan, int lane,
                                        uint64_t *full_bar, uint64_t *empty_bar, uint32_t *issued,
                                        volatile int *abort_flag, Issue issue) {
  grid_dependency_wait();
  long long e = 0;
  bool aborted = false;
#ifdef PA_TRACE
  long long tr_t0 = clock64(), tr_tab = 0, tr_empty = 0, tr_segs = 0;
#endif
  for (int ph = 0; ph < 2 && !aborted; ++ph) {
    long long from, to;
    if (!phase_range(plan, ph, &from, &to)) continue;
    Walk wk;
    if (ph == 0)
      wk.start(a, plan.sA, plan.rA, from, plan.cA);
    else
      wk.start(a, plan.s0, plan.r0, from, plan.c0);
    while (wk.w < to && !aborted) {
      const int n = wk.seg_len(to);
      const int kvh = wk.pc / HC;
      const int L = wk.L;
      const int32_t *trow = a.tables + (long long)wk.s * a.max_blocks + wk.b;
      int pid_next = lane < n ? trow[lane] : -1;
#ifdef PA_TRACE
      {
        const long long t = clock64();
        pid_next = __shfl_sync(kFullMask, pid_next, lane);  // wait for the table load
        tr_tab += clock64() - t;
        ++tr_segs;
      }
#endif
      for (int base = 0; base < n && !aborted; base += 32) {
        const int pid_cur = pid_next;
        const int cnt = min(32, n - base);
        if (base + 32 < n) pid_next = (base + 32 + lane < n) ? trow[base + 32 + lane] : -1;
        for (int k = 0; k < cnt; k += a.pg) {
          const int t = k + lane;
          const int p = __shfl_sync(kFullMask, pid_cur, t < 32 ? t : 31);
          bool fail = false;
          if (lane < a.pg && t < cnt) {
            const uint32_t me = uint32_t(e) + uint32_t(lane);  // a CTA's entry count fits 32 bits
            const int slot = int(me % uint32_t(a.nstage));
            const uint32_t u = me / uint32_t(a.nstage);
#ifdef PA_TRACE
            const long long t = clock64();
#endif
            if (*abort_flag || (u > 0 && !mbar_wait(&empty_bar[slot], (u - 1) & 1u, abort_flag))) {
              fail = true;
            } else {
#ifdef PA_TRACE
              if (lane == 0) tr_empty += clock64() - t;
#endif
#ifdef PA_FAULT_WITHHOLD_FIRST_ENTRY
              // Test build only: the first entry of the CTA whose range starts
              // at the step's first tile is never issued (no copy and no
              // arrival), so the consumer that waits for it runs into its wait
              // limit, as a lost arrival would make it.
              const bool withhold = plan.w0 == 0 && me == 0;
#else
              constexpr bool withhold = false;
#endif
              if (!withhold) {
                issue(slot, p, kvh, wk.b + base + t, L, wk.s, wk.pc, base + t < a.ncw);
                issued[slot] = u + 1;
              }
            }
          }
          if (__any_sync(kFullMask, fail)) {
            aborted = true;
            if (lane == 0) {
              *abort_flag = 1;
              raise_error(a.err, PA_DEVERR_TIMEOUT);
            }
            break;
          }
          e += min(a.pg, cnt - k);
        }
      }
      wk.advance(a, n, PC);
    }
  }
#ifdef PA_TRACE
  if (lane == 0 && PA_TRACE_CTA(blockIdx.x))
    printf("trace cta %d producer: segments %lld cycles %lld table-wait %lld slot-wait(lane0) %lld\n", blockIdx.x,
           tr_segs, clock64() - tr_t0, tr_tab, tr_empty);
#endif
  // Do not leave while a copy into this CTA's shared memory is in flight:
  // only the last use issued into a slot can be (earlier ones were released,
  // which needs them landed).
  __syncwarp();
  if (lane == 0) {
    for (int slot = 0; slot < a.nstage; ++slot) {
      if (issued[slot] == 0) continue;
      int never = 0;
      mbar_wait(&full_bar[slot], (issued[slot] - 1) & 1u, &never);
    }
  }
}

// Consumer warps that take at least one tile of the segment [j, j + n) of a
// CTA's processing order (tile j goes to warp j % ncw), as a bit mask.
__device__ __forceinline__ unsigned participants(long long j, int n, int ncw) {
  if (n >= ncw) return (1u << ncw) - 1u;
  const int w0 = int(uint32_t(j) % uint32_t(ncw));  // a CTA's tile count fits 32 bits
  const unsigned run = (1u << n) - 1u;
  return ((run << w0) | (run >> (ncw - w0))) & ((1u << ncw) - 1u);
}

// Zero output rows of the sequences with nothing to read, spread over CTAs.
template <typename T>
__device__ __forceinline__ void zero_empty_rows(const DecodeArgs &a, int D, int tid, int nthreads) {
  for (int s = blockIdx.x; s < a.S; s += a.nctas) {
    if (eff_len(a, s) != 0) continue;
    for (int i = tid; i < a.Hq * D; i += nthreads) store_out1<T>(a, (long long)s * a.Hq + i / D, i % D, D, 0.f);
  }
}

// Floats per head in a warp state or a partial record: acc[D], m, l, and two
// pad floats so that every head row starts on a 16-byte boundary.
__host__ __device__ constexpr int state_row(int D) { return D + 4; }

// The merger warp.  It walks the same plan as the consumers, one segment at
// a time.  Only the consumer warps that took a tile of a segment (the
// participants) hand it a state: warp w deposits (acc[D], m, l per head; head
// stride state_row(D), warp stride warp_stride) in its own buffer of `mrg` and
// arrives on st_full[w]; the merger waits for the participants, combines
//     M = max_w m_w;  num = sum_w 2^(m_w - M) acc_w;  den = sum_w 2^(m_w - M) l_w,
// and writes num / den as the output rows (the segment is a whole (s, pc)) or
// this CTA's partial record (num, M, den) for a (s, pc) cut by a range
// boundary, then hands each buffer back (st_free[w]).  Each warp has its own
// pair of barriers, so warps never wait for one another's segments: a run of
// one-tile segments (short sequences) spreads over the four warps.  With
// kSoloWrites, a whole (s, pc) taken by a single warp is normalised and
// written by that warp and never reaches the merger.  For a cut (s, pc) the
// merger counts this CTA in; the CTA that completes the count merges the
// records of all CTAs that share the pair (the a5 step) and sets the counter
// back to zero:
//     M = max_r m_r;  out = sum_r 2^(m_r - M) acc_r / sum_r 2^(m_r - M) l_r.
// Running this off the consumer warps keeps every fence, atomic and remote
// read of a segment end out of the streaming path.  The weights are formed
// once per (warp or record, head); the rows then move as 16-byte vectors, so
// a merge costs one L2 round trip per record rather than one per element.
template <typename T, int D, bool kSoloWrites>
__device__ __forceinline__ void run_merger(const DecodeArgs &a, const Plan &plan, int PC, int HC, int G, int lane,
                                           const float *mrg, int warp_stride, int nbuf, uint64_t *st_full,
                                           uint64_t *st_free, float *sh_w, volatile int *abort_flag) {
  constexpr int R = state_row(D);
  constexpr int C4 = D / 4;            // 16-byte chunks per head row
  constexpr int kIters = 8 * C4 / 32;  // chunks per lane for 8 heads
  static_assert(kConsumerWarps == 4 && (8 * C4) % 32 == 0, "lane = 4 * head + warp below");
  const int GT = a.GT;
  const int N = a.nctas;
  const long long Wc = plan.Wc;
  const int lh = lane >> 2, lq = lane & 3;  // the (head, warp) whose weight this lane forms
  float *sh_m = sh_w, *sh_l = sh_w + kMergeRecords * 8;
  int *sh_rec = reinterpret_cast<int *>(sh_w + 2 * kMergeRecords * 8);  // contributors of a cut pair
  long long k = 0;  // segments handled
  long long j = 0;  // tiles before the current segment, in processing order
  uint32_t taken[kConsumerWarps] = {0u, 0u, 0u, 0u};  // deposits taken from each warp
#ifdef PA_TRACE
  long long tr_t0 = clock64(), tr_wait = 0, tr_comb = 0, tr_cut = 0, tr_adv = 0, tr_solo = 0, tr_c = 0;
#endif
  for (int ph = 0; ph < 2; ++ph) {
    long long from, to;
    if (!phase_range(plan, ph, &from, &to)) continue;
    Walk wk;
    if (ph == 0)
      wk.start(a, plan.sA, plan.rA, from, plan.cA);
    else
      wk.start(a, plan.s0, plan.r0, from, plan.c0);
    while (wk.w < to) {
      const int n = wk.seg_len(to);
      const bool complete = (wk.b == 0 && n == wk.nb);
      const bool first_seg = (wk.w == plan.w0);
      const int s = wk.s, pc = wk.pc;
      const int hq0 = (pc / HC) * G + (pc % HC) * GT;
#ifdef PA_TRACE
      const long long tr_w0 = clock64();
#endif
      const unsigned pm = participants(j, n, a.ncw);
      if (kSoloWrites && complete && __popc(pm) == 1) {  // the warp wrote the rows itself
        j += n;
        wk.advance(a, n, PC);
#ifdef PA_TRACE
        tr_solo += clock64() - tr_w0;
#endif
        continue;
      }
#pragma unroll
      for (int q = 0; q < kConsumerWarps; ++q) {
        const uint32_t bq = nbuf == 2 ? (taken[q] & 1u) : 0u, uq = nbuf == 2 ? (taken[q] >> 1) : taken[q];
        if (((pm >> q) & 1u) && !mbar_wait(&st_full[2 * q + bq], uq & 1u, abort_flag)) {
          if (lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
      }
#ifdef PA_TRACE
      tr_wait += clock64() - tr_w0;
      tr_c = clock64();
#endif
      __syncwarp();
      // ---- combine the participants' states: weights per (warp, head) ...
      const bool mine = lh < GT && ((pm >> lq) & 1u);
      // the buffer each warp's state of this segment is in (head slots 4 b ..)
      int boff[kConsumerWarps];
#pragma unroll
      for (int q = 0; q < kConsumerWarps; ++q) boff[q] = nbuf == 2 ? int(taken[q] & 1u) * 4 * R : 0;
      const int boff_l = lq == 0 ? boff[0] : lq == 1 ? boff[1] : lq == 2 ? boff[2] : boff[3];
      float m = -CUDART_INF_F, l = 0.f;
      if (mine) {
        m = mrg[lq * warp_stride + boff_l + lh * R + D];
        l = mrg[lq * warp_stride + boff_l + lh * R + D + 1];
      }
      float M = fmaxf(m, __shfl_xor_sync(kFullMask, m, 1));
      M = fmaxf(M, __shfl_xor_sync(kFullMask, M, 2));
      const float f = mine ? fast_exp2(m - M) : 0.f;
      float den = f * l;
      den += __shfl_xor_sync(kFullMask, den, 1);
      den += __shfl_xor_sync(kFullMask, den, 2);
      const float wt = complete ? (mine ? f / den : 0.f) : f;
      float *rec = nullptr;
      if (!complete) {
        long long ro = ((long long)blockIdx.x * 2 + (first_seg ? 0 : 1)) * 8 * R;
        PA_DBG_FIX(ro >= 0 && ro + 8 * R <= (long long)N * 2 * 8 * R, kDbgGlobal, ro = 0);
        rec = a.partials + ro;
        if (lq == 0 && lh < GT) {
          rec[lh * R + D] = M;
          rec[lh * R + D + 1] = den;
        }
      }
      // ... then the rows, 4 floats per lane and step, over the chunks of the
      // GT heads only (one step per head at D = 128: one step on an MHA layer)
#pragma unroll
      for (int i = 0; i < kIters; ++i) {
        if (32 * i >= GT * C4) break;
        const int c = lane + 32 * i;
        const int h = c / C4, d = (c % C4) * 4;
        float w[kConsumerWarps];
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q) w[q] = __shfl_sync(kFullMask, wt, 4 * h + q);
        if (h < GT) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kConsumerWarps; ++q) {
            if (!((pm >> q) & 1u)) continue;  // a buffer that got no state this segment
            const float4 v = *reinterpret_cast<const float4 *>(mrg + q * warp_stride + boff[q] + h * R + d);
            acc.x += w[q] * v.x;
            acc.y += w[q] * v.y;
            acc.z += w[q] * v.z;
            acc.w += w[q] * v.w;
          }
          if (complete) {
            long long orow = (long long)s * a.Hq + hq0 + h;
            PA_DBG_FIX(orow >= 0 && orow < (long long)a.S * a.Hq, kDbgGlobal, orow = 0);
            store_out4<T>(a, orow, d, D, acc);
          } else {
            *reinterpret_cast<float4 *>(rec + h * R + d) = acc;
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < kConsumerWarps; ++q) {
        if ((pm >> q) & 1u) {
          if (lane == 0) mbar_arrive(&st_free[2 * q + (nbuf == 2 ? (taken[q] & 1u) : 0u)]);  // warp q may reuse it now
          ++taken[q];
        }
      }
#ifdef PA_TRACE
      tr_comb += clock64() - tr_c;
      tr_c = clock64();
#endif
      if (!complete) {
        // ---- count this CTA in; the last of the pair's CTAs merges
        __syncwarp();  // every lane's record writes come before lane 0's release below
        // the pair's tiles sit at cost positions Cp + kSegCost + b, b < nb
        const long long Cp = wk.cp;
        const int nb = wk.nb;
        const int cf = cta_at_cost(Cp + kSegCost, Wc, N);
        const int cl = cta_at_cost(Cp + kSegCost + nb - 1, Wc, N);
        // a CTA strictly between cf and cl owns tiles of the pair iff its cost
        // range holds a position (always when Wc >= N)
        auto owns = [&](int c) { return c == cf || c == cl || cost_start(c, Wc, N) < cost_start(c + 1, Wc, N); };
        // the pair's contributors: the CTAs of [cf, cl] that own tiles of it,
        // found 32 at a time; the first kMergeRecords are listed in sh_rec
        int kc = 0;
        if (Wc >= N) {
          kc = cl - cf + 1;
          for (int r = lane; r < min(kc, kMergeRecords); r += 32) sh_rec[r] = cf + r;
        } else {
          for (int base = cf; base <= cl; base += 32) {
            const int c = base + lane;
            const bool has = c <= cl && owns(c);
            const unsigned mk = __ballot_sync(kFullMask, has);
            const int pos = kc + __popc(mk & ((1u << lane) - 1u));
            if (has && pos < kMergeRecords) sh_rec[pos] = c;
            kc += __popc(mk);
          }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          // release this CTA's record; the last contributor also acquires the
          // records the others released before their counts
          unsigned *ctr = a.counters + (long long)s * PC + pc;
          const unsigned seen = atomic_add_acq_rel_gpu(ctr, 1u) + 1u;
          last = seen == unsigned(kc);
          if (last) *ctr = 0u;  // ready for the next call
        }
        last = __shfl_sync(kFullMask, last, 0);
        __syncwarp();  // the other lanes' record reads come after lane 0's acquire
        if (last) {
          // the pair is cf's last segment iff cf also owns the tile before it (at Cp - 1)
          const bool cf_last_seg = Cp > 0 && cta_at_cost(Cp - 1, Wc, N) == cf;
          auto rec_of = [&](int c) {
            const int slot = (c == cf && cf_last_seg) ? 1 : 0;
            return a.partials + ((long long)c * 2 + slot) * 8 * R;
          };
          const int nrec = kc;
          if (nrec <= 2) {
            // the common cut: a pair split between two CTAs.  Both records'
            // rows (GT heads) and their (m, l) in one batch of L2 reads, then
            // the weights and the combine in registers.
            const float *ra = rec_of(sh_rec[0]);
            const float *rb = nrec == 2 ? rec_of(sh_rec[1]) : ra;
            float4 va[kIters], vb[kIters];
#pragma unroll
            for (int i = 0; i < kIters; ++i) {
              va[i] = vb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              const int c = lane + 32 * i;
              const int h = c / C4, d = (c % C4) * 4;
              if (32 * i < GT * C4 && h < GT) {
                va[i] = __ldcg(reinterpret_cast<const float4 *>(ra + h * R + d));
                if (nrec == 2) vb[i] = __ldcg(reinterpret_cast<const float4 *>(rb + h * R + d));
              }
            }
            // lane hh + 8 rs holds (m, l) of record rs for head hh
            const int hh = lane & 7, rs = lane >> 3;
            const bool has = hh < GT && rs < nrec;
            const float *rr = (rs == 0 ? ra : rb) + hh * R;
            const float mv = has ? __ldcg(rr + D) : -CUDART_INF_F;
            const float lv = has ? __ldcg(rr + D + 1) : 0.f;
            const float Mh = fmaxf(mv, __shfl_xor_sync(kFullMask, mv, 8));
            const float fv = has ? fast_exp2(mv - Mh) : 0.f;
            float den = fv * lv;
            den += __shfl_xor_sync(kFullMask, den, 8);
            const float wv = has ? fv / den : 0.f;  // weight of record rs for head hh
#pragma unroll
            for (int i = 0; i < kIters; ++i) {
              if (32 * i >= GT * C4) break;
              const int c = lane + 32 * i;
              const int h = c / C4, d = (c % C4) * 4;
              const float wa = __shfl_sync(kFullMask, wv, h & 7), wb = __shfl_sync(kFullMask, wv, 8 + (h & 7));
              if (h < GT) {
                float4 o;
                o.x = wa * va[i].x + wb * vb[i].x;
                o.y = wa * va[i].y + wb * vb[i].y;
                o.z = wa * va[i].z + wb * vb[i].z;
                o.w = wa * va[i].w + wb * vb[i].w;
                store_out4<T>(a, (long long)s * a.Hq + hq0 + h, d, D, o);
              }
            }
          } else if (nrec <= kMergeRecords) {
            // every record's (m, l) per head at once, then the weights
            //     2^(m_r - M) / sum_r 2^(m_r - M) l_r   (in place of m_r)
            for (int i = lane; i < nrec * GT; i += 32) {
              const int r = i / GT, h = i - r * GT;
              const float *rr = rec_of(sh_rec[r]) + h * R;
              sh_m[r * 8 + h] = __ldcg(rr + D);
              sh_l[r * 8 + h] = __ldcg(rr + D + 1);
            }
            __syncwarp();
            if (lane < GT) {
              const int h = lane;
              float Mr = -CUDART_INF_F;
              for (int r = 0; r < nrec; ++r) Mr = fmaxf(Mr, sh_m[r * 8 + h]);
              float dr = 0.f;
              for (int r = 0; r < nrec; ++r) {
                const float fr = fast_exp2(sh_m[r * 8 + h] - Mr);
                sh_m[r * 8 + h] = fr;
                dr += fr * sh_l[r * 8 + h];
              }
              const float inv = 1.f / dr;
              for (int r = 0; r < nrec; ++r) sh_m[r * 8 + h] *= inv;
            }
            __syncwarp();
            float4 acc[kIters];
#pragma unroll
            for (int i = 0; i < kIters; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < nrec; ++r) {
              const float *rr = rec_of(sh_rec[r]);
#pragma unroll
              for (int i = 0; i < kIters; ++i) {
                const int c = lane + 32 * i;
                const int h = c / C4, d = (c % C4) * 4;
                if (h < GT) {
                  const float wr = sh_m[r * 8 + h];
                  const float4 v = __ldcg(reinterpret_cast<const float4 *>(rr + h * R + d));
                  acc[i].x += wr * v.x;
                  acc[i].y += wr * v.y;
                  acc[i].z += wr * v.z;
                  acc[i].w += wr * v.w;
                }
              }
            }
#pragma unroll
            for (int i = 0; i < kIters; ++i) {
              const int c = lane + 32 * i;
              const int h = c / C4, d = (c % C4) * 4;
              if (h < GT) store_out4<T>(a, (long long)s * a.Hq + hq0 + h, d, D, acc[i]);
            }
            __syncwarp();  // sh_m / sh_l / sh_rec are reused by the next merge
          } else {
            // more than kMergeRecords contributors: per element, straight from the records
            for (int idx = lane; idx < GT * D; idx += 32) {
              const int h = idx / D;
              const int d = idx - h * D;
              float Mr = -CUDART_INF_F;
              for (int c = cf; c <= cl; ++c) {
                if (!owns(c)) continue;
                Mr = fmaxf(Mr, __ldcg(rec_of(c) + h * R + D));
              }
              float num = 0.f, dr = 0.f;
              for (int c = cf; c <= cl; ++c) {
                if (!owns(c)) continue;
                const float *rr = rec_of(c) + h * R;
                const float fr = fast_exp2(__ldcg(rr + D) - Mr);
                num += fr * __ldcg(rr + d);
                dr += fr * __ldcg(rr + D + 1);
              }
              store_out1<T>(a, (long long)s * a.Hq + hq0 + h, d, D, num / dr);
            }
          }
        }
      }
#ifdef PA_TRACE
      tr_cut += clock64() - tr_c;
      tr_c = clock64();
#endif
      ++k;
      j += n;
      wk.advance(a, n, PC);
#ifdef PA_TRACE
      tr_adv += clock64() - tr_c;
#endif
    }
  }
#ifdef PA_TRACE
  if (lane == 0 && PA_TRACE_CTA(blockIdx.x))
    printf("trace cta %d merger: segments %lld cycles %lld waiting %lld combine %lld cut %lld advance %lld solo %lld\n",
           blockIdx.x, k, clock64() - tr_t0, tr_wait, tr_comb, tr_cut, tr_adv, tr_solo);
#endif
}

// A consumer warp's hand-off of its state for a segment it took tiles of:
// wait until the merger took this warp's previous deposit (its st_free, phase
// dep - 1: the merger frees one warp's deposits in order, so the parity test
// is exact), then let `write` store the state into the warp's buffer and
// announce it (its st_full).
template <class Write>
__device__ __forceinline__ void deposit_state(const DecodeArgs &a, long long use, int lane, uint64_t *st_full,
                                              uint64_t *st_free, volatile int *abort_flag, Write write) {
  // `use`: how many states this warp has put in this buffer before
  if (use > 0 && !mbar_wait(st_free, uint32_t(use - 1) & 1u, abort_flag)) {
    if (lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  __syncwarp();
  write();
  __syncwarp();
  if (lane == 0) mbar_arrive(st_full);
}

}  // namespace pagedkv
