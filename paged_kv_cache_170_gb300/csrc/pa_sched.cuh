// pa_sched.cuh -- work schedule shared by the two decode kernels.
//
// The step's work is the ordered list of tiles (sequence s, pair-chunk pc,
// logical block b), pc = kv head * HC + head chunk, where a head chunk is GT
// of the G query heads that share one kv head and a tile is one physical
// block of K plus the same block of V for that kv head.  The W tiles are cut
// into N equal contiguous ranges, one per CTA (N = one full wave, 2 CTAs per
// SM): every CTA streams the same number of bytes whatever the length mix.
// A CTA finishes any (s, pc) whose tiles all fall in its range and writes
// `out`; a (s, pc) cut by a range boundary leaves a partial (acc, m, l) for
// the reduce kernel: slot 0 for the CTA's first segment, slot 1 for its last.
#pragma once

#include <math_constants.h>

#include "pa_common.cuh"

namespace pagedkv {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kCtasPerSm = 2;
constexpr int kMaxStages = 64;
constexpr int kMaxBlockSize = 64;
constexpr int kRingBytes = 80 * 1024;

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
  float *partials;         // [N][2][GT][D + 2]: acc[D], m, l
  long long *cum;          // [S + 1] tile prefix (written by CTA 0)
  int *err;
  int nctas;
  int nstage;
  uint32_t slot_stride;    // bytes between ring slots (one slot = K tile + V tile)
  uint32_t tile_stride;    // offset of the V tile inside a slot
  int GT;                  // query heads per pair-chunk (<= 8)
  int ncw;                 // consumer warps that take tiles
  int pg;                  // ring entries the producer issues at once (ncw + pg <= nstage)
  int nops;                // tensor copies per tile (1: one 3-D box; 2: two 2-D halves)
};

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
__device__ __forceinline__ bool wait_entry(uint64_t *full, uint64_t *empty, long long e, int nstage,
                                           volatile int *abort) {
  const int slot = int(e % nstage);
  const uint32_t u = uint32_t(e / nstage);
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

__device__ __forceinline__ int blocks_of(const DecodeArgs &a, int s) {
  return (clamped_len(a, s) + a.B - 1) / a.B;
}

// Total tile count W (and, in CTA 0, the per-sequence prefix) and the tile
// where this CTA's range starts.  Run by one whole warp.
__device__ __forceinline__ void schedule_scan(const DecodeArgs &a, int PC, int lane, long long *W_out,
                                              int *s0_out, long long *r0_out) {
  const int cap = a.max_blocks * a.B;
  long long run = 0;
  for (int base = 0; base < a.S; base += 32) {
    const int s = base + lane;
    long long n = 0;
    if (s < a.S) {
      const int L = a.lens[s];
      if ((L < 0 || L > cap) && blockIdx.x == 0) raise_error(a.err, PA_DEVERR_CONTEXT);
      n = (long long)blocks_of(a, s) * PC;
    }
    long long incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += y;
    }
    if (blockIdx.x == 0 && s < a.S) a.cum[s] = run + incl - n;
    run += __shfl_sync(kFullMask, incl, 31);
  }
  if (blockIdx.x == 0 && lane == 0) a.cum[a.S] = run;
  const long long W = run;
  const long long w0 = (long long)blockIdx.x * W / a.nctas;
  int s0 = a.S;
  long long r0 = 0;
  run = 0;
  for (int base = 0; base < a.S && s0 == a.S; base += 32) {
    const int s = base + lane;
    const long long n = s < a.S ? (long long)blocks_of(a, s) * PC : 0;
    long long incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += y;
    }
    const long long excl = run + incl - n;
    const bool hit = n > 0 && excl <= w0 && w0 < run + incl;
    const unsigned m = __ballot_sync(kFullMask, hit);
    if (m) {
      const int leader = __ffs(m) - 1;
      s0 = __shfl_sync(kFullMask, s, leader);
      r0 = __shfl_sync(kFullMask, w0 - excl, leader);
    }
    run += __shfl_sync(kFullMask, incl, 31);
  }
  *W_out = W;
  *s0_out = s0;
  *r0_out = r0;
}

// Cursor over a CTA's tile range, one segment (consecutive tiles of one
// (s, pc)) at a time.  Producer and consumers walk identical sequences.
struct Walk {
  int s, pc, b, nb;
  long long w;
  __device__ __forceinline__ void start(const DecodeArgs &a, int s0, long long r0, long long w0) {
    s = s0;
    nb = blocks_of(a, s);
    pc = int(r0 / nb);
    b = int(r0 % nb);
    w = w0;
  }
  __device__ __forceinline__ int seg_len(long long w1) const {
    return int((long long)(nb - b) < w1 - w ? (long long)(nb - b) : w1 - w);
  }
  __device__ __forceinline__ void advance(const DecodeArgs &a, int n, int PC) {
    w += n;
    b += n;
    if (b == nb) {
      b = 0;
      if (++pc == PC) {
        pc = 0;
        do {
          ++s;
        } while (s < a.S && blocks_of(a, s) == 0);
        if (s < a.S) nb = blocks_of(a, s);
      }
    }
  }
};

// The producer warp: walks the CTA's range, reads the block table 32 entries
// at a time (coalesced, next batch prefetched, kept in registers: never
// re-read per token) and fills the ring.  Entries are issued in groups of pg:
// lane i < pg claims entry e + i (waits until its slot's previous use was
// released) and calls issue(slot, pid, kv head, logical block, context len),
// which announces the bytes on full_bar[slot] and starts the copies; the lanes
// of a group wait and issue in parallel.  issued[slot] keeps the last use
// issued into each slot so the producer can wait for every copy still in
// flight before it leaves (after an abort too).
template <class Issue>
__device__ __forceinline__ void produce(const DecodeArgs &a, int PC, int HC, int s0, long long r0, long long w0,
                                        long long w1, int lane, uint64_t *full_bar, uint64_t *empty_bar,
                                        uint32_t *issued, volatile int *abort_flag, Issue issue) {
  long long e = 0;
  bool aborted = false;
  Walk wk;
  wk.start(a, s0, r0, w0);
  while (wk.w < w1 && !aborted) {
    const int n = wk.seg_len(w1);
    const int kvh = wk.pc / HC;
    const int L = clamped_len(a, wk.s);
    const int32_t *trow = a.tables + (long long)wk.s * a.max_blocks + wk.b;
    int pid_next = lane < n ? trow[lane] : -1;
    for (int base = 0; base < n && !aborted; base += 32) {
      const int pid_cur = pid_next;
      const int cnt = min(32, n - base);
      if (base + 32 < n) pid_next = (base + 32 + lane < n) ? trow[base + 32 + lane] : -1;
      for (int k = 0; k < cnt; k += a.pg) {
        const int t = k + lane;
        const int p = __shfl_sync(kFullMask, pid_cur, t < 32 ? t : 31);
        bool fail = false;
        if (lane < a.pg && t < cnt) {
          const long long me = e + lane;
          const int slot = int(me % a.nstage);
          const uint32_t u = uint32_t(me / a.nstage);
          if (*abort_flag || (u > 0 && !mbar_wait(&empty_bar[slot], (u - 1) & 1u, abort_flag))) {
            fail = true;
          } else {
            issue(slot, p, kvh, wk.b + base + t, L);
            issued[slot] = u + 1;
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

// Merge the consumer warps' states of one segment, held in shared memory as
// mrg[warp][head][0..D-1 acc, D: m, D+1: l] (head stride D + 2), and write the
// final rows (segment covers the whole (s, pc)) or this CTA's partial record.
template <typename T>
__device__ __forceinline__ void combine_segment(const DecodeArgs &a, const float *mrg, int warp_stride, int D,
                                                int GT, bool complete, bool first_seg, int s, int hq0, int tid,
                                                int nthreads) {
  for (int idx = tid; idx < GT * D; idx += nthreads) {
    const int h = idx / D;
    const int d = idx - h * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int q = 0; q < kConsumerWarps; ++q) M = fmaxf(M, mrg[q * warp_stride + h * (D + 2) + D]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int q = 0; q < kConsumerWarps; ++q) {
      const float *row = mrg + q * warp_stride + h * (D + 2);
      const float f = fast_exp2(row[D] - M);
      num += f * row[d];
      den += f * row[D + 1];
    }
    if (complete) {
      long long oo = ((long long)s * a.Hq + hq0 + h) * D + d;
      PA_DBG_FIX(oo >= 0 && oo < (long long)a.S * a.Hq * D, kDbgGlobal, continue);
      T *o = static_cast<T *>(a.out) + oo;
      *o = Elem<T>::from_float(num / den);
    } else {
      long long ro = (((long long)blockIdx.x * 2 + (first_seg ? 0 : 1)) * GT + h) * (D + 2);
      PA_DBG_FIX(ro >= 0 && ro + D + 2 <= (long long)a.nctas * 2 * 8 * (D + 2), kDbgGlobal, continue);
      float *rec = a.partials + ro;
      rec[d] = num;
      if (d == 0) {
        rec[D] = M;
        rec[D + 1] = den;
      }
    }
  }
}

}  // namespace pagedkv
