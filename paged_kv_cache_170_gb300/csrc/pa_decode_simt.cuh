// pa_decode_simt.cuh -- split-context paged decode kernel on CUDA cores (a4):
// the path for fp32 caches and block sizes that are not a multiple of 16.
//
// Work decomposition.  The step's work is the ordered list of tiles
// (sequence s, pair-chunk pc, logical block b), pc = kv head * HC + head
// chunk, where a head chunk is GT of the G query heads that share one kv head
// and a tile is one physical block of K plus the same block of V for that kv
// head (B*D contiguous elements each).  The W tiles are cut into N equal
// contiguous ranges, one per CTA, N = one full wave (2 CTAs per SM): every
// CTA streams the same number of bytes whatever the length mix, so no SM
// idles at the tail.  A CTA finishes any (s, pc) whose tiles all fall in its
// range and writes `out`; a (s, pc) cut by a range boundary leaves a partial
// (m, l, acc) for the reduce kernel.
//
// Inside a CTA.  One producer warp walks the range in order, reads the block
// table once per 32 tiles (coalesced, kept in registers: the table is never
// re-read per token), and fills a ring of shared-memory slots, one slot per
// (block, kv head): lanes 0 and 1 issue the 1-D bulk copies (TMA) of the K
// tile and of the V tile in one instruction, completion counted in bytes on
// the slot's mbarrier.  Only the valid rows of a sequence's last, partly
// filled block are copied.  Four consumer warps take tiles round-robin; each keeps its own
// running max / sum / accumulator (online softmax, base 2) and the four
// states are merged when the (s, pc) ends.
//
// Per tile and consumer warp (fp32 arithmetic, packed fma.rn.f32x2):
//   QK: a token is handled by LPT lanes, each owning DPL dimensions of every
//       query head of the chunk (q pre-scaled by scale*log2(e), in registers);
//       the partial dots are summed across the LPT lanes with xor shuffles.
//   softmax: tile max per head (shuffles), rescale of the running state,
//       p = 2^(x - m) written to a per-warp score buffer.
//   PV: lanes own D/32 dimensions; every token's p's are broadcast from the
//       score buffer and accumulated for all GT heads.
#pragma once

#include "pa_sched.cuh"

namespace pagedkv {

template <typename T, int D, int GT>
struct DecodeCfg {
  static constexpr int EPC = 16 / int(sizeof(T));                 // elements per 16-byte chunk
  static constexpr int DPL = (D == 128 && GT <= 4) ? 16 : 8;      // dims per lane in QK
  static constexpr int LPT = D / DPL;                             // lanes per token in QK
  static constexpr int TS = 32 / LPT;                             // tokens per QK pass
  static constexpr int CPL = DPL / EPC;                           // 16-byte chunks per lane per token
  static constexpr int DPV = D / 32;                              // dims per lane in PV
  static_assert(DPL % EPC == 0, "lane slice must be whole chunks");
  static_assert(LPT >= 8, "a quarter warp must read one contiguous 128-byte run");
  static_assert(GT <= LPT, "one score per lane");
};

// V row slice of a lane: DPV elements starting at dimension lane * DPV.
template <typename T, int DPV>
__device__ __forceinline__ void load_v(const char *row, int lane, float2 *vf) {
  const char *p = row + size_t(lane) * DPV * sizeof(T);
  if constexpr (sizeof(T) == 4 && DPV == 4) {
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    Elem<float>::chunk_to_f2(r, vf);
  } else if constexpr (sizeof(T) == 4 && DPV == 2) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    vf[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
  } else if constexpr (sizeof(T) == 2 && DPV == 4) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    vf[0] = Elem<T>::word_to_f2(r.x);
    vf[1] = Elem<T>::word_to_f2(r.y);
  } else {
    static_assert(sizeof(T) == 2 && DPV == 2, "unsupported V slice");
    vf[0] = Elem<T>::word_to_f2(*reinterpret_cast<const uint32_t *>(p));
  }
}

// The GT probabilities of token t from the warp's score buffer.
template <int GT>
__device__ __forceinline__ void load_p(const float *sc, int t, float *p) {
  if constexpr (GT == 8) {
    const float4 a = *reinterpret_cast<const float4 *>(sc + t * 8);
    const float4 b = *reinterpret_cast<const float4 *>(sc + t * 8 + 4);
    p[0] = a.x; p[1] = a.y; p[2] = a.z; p[3] = a.w; p[4] = b.x; p[5] = b.y; p[6] = b.z; p[7] = b.w;
  } else if constexpr (GT == 4) {
    const float4 a = *reinterpret_cast<const float4 *>(sc + t * 4);
    p[0] = a.x; p[1] = a.y; p[2] = a.z; p[3] = a.w;
  } else if constexpr (GT == 2) {
    const float2 a = *reinterpret_cast<const float2 *>(sc + t * 2);
    p[0] = a.x; p[1] = a.y;
  } else {
    p[0] = sc[t];
  }
}

template <typename T, int D, int GT>
__global__ void __launch_bounds__(kDecodeThreads, kCtasPerSm) decode_partition_kernel(const DecodeArgs a) {
  using C = DecodeCfg<T, D, GT>;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(16) float sc_buf[kConsumerWarps][kMaxBlockSize * GT];
  __shared__ __align__(16) float mrg[kConsumerWarps][GT][state_row(D)];
  __shared__ Plan sh_plan;
  __shared__ uint32_t issued[kMaxStages];
  __shared__ int sh_abort;
  // hand-off of mrg[w] (one buffer here; the [2] layout is the merger's)
  __shared__ __align__(8) uint64_t st_full[kConsumerWarps][2], st_free[kConsumerWarps][2];
  __shared__ float sh_mw[kMergeScratch];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int HC = G / GT;
  const int PC = a.Hkv * HC;
  const int B = a.B;
  volatile int *abort_flag = &sh_abort;

#ifdef PA_TRACE
  __shared__ unsigned long long tr_start;
  if (threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tr_start));
#endif
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nstage; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
      issued[i] = 0;
    }
    for (int w = 0; w < kConsumerWarps; ++w) {
      mbar_init(&st_full[w][0], 1);
      mbar_init(&st_free[w][0], 1);
    }
    sh_abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp) {
    Plan plan;
    schedule_scan(a, PC, lane, &plan);
    if (lane == 0) {
      sh_plan = plan;
    }
  }
  __syncthreads();

  const Plan plan = sh_plan;
  const long long w0 = plan.w0, w1 = plan.w1;
  if (w0 >= w1) {  // fewer tiles than CTAs: nothing to stream, only empty rows to zero
    if (warp == kMergerWarp) zero_empty_rows<T>(a, D, lane, 32);
    if (warp == kProducerWarp) grid_dependency_wait();  // never complete before the grid this one depends on
    return;
  }
  const size_t tile_elems = size_t(B) * D;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    produce(a, PC, HC, plan, lane, full_bar, empty_bar, issued, abort_flag,
            [&](int slot, int p, int kvh, int bb, int L, int, int, bool) {
              if (p < 0 || p >= a.num_blocks) {
                raise_error(a.err, PA_DEVERR_BLOCK_ID);
                mbar_arrive(&full_bar[slot]);  // complete the phase without data
                return;
              }
              const int nv = min(B, L - bb * B);
              const uint32_t bytes = uint32_t(nv) * D * sizeof(T);  // valid rows only
              const size_t off = ((size_t)p * a.Hkv + kvh) * tile_elems * sizeof(T);
              mbar_arrive_expect_tx(&full_bar[slot], 2 * bytes);
              unsigned char *dst = ring + size_t(slot) * a.slot_stride;
              bulk_g2s(dst, a.k_cache + off, bytes, &full_bar[slot]);
              bulk_g2s(dst + a.tile_stride, a.v_cache + off, bytes, &full_bar[slot]);
            });
    return;
  }

  if (warp == kMergerWarp) {
    // -------------------------------------------------------------- merger
    run_merger<T, D, false>(a, plan, PC, HC, G, lane, &mrg[0][0][0], GT * state_row(D), 1, &st_full[0][0],
                            &st_free[0][0], sh_mw,
                            abort_flag);
    zero_empty_rows<T>(a, D, lane, 32);
#ifdef PA_TRACE
    if (lane == 0) {
      unsigned long long t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      printf("tracet %d %u %llu %llu %lld\n", blockIdx.x, 0u, tr_start, t1, w1 - w0);
    }
#endif
    return;
  }

  // -------------------------------------------------------------- consumers
  float *sc = sc_buf[warp];
  const int jl = lane % C::LPT;   // lane within its token group (QK)
  const int tsub = lane / C::LPT; // token slot of the lane (QK)
  // Softmax state (m_mine, l_mine) of a lane belongs to head lane % GT.

  long long j = 0;      // tiles, in this CTA's processing order
  long long dep = 0;    // states this warp deposited for the merger
  // rotated processing order (see Plan)
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
      const int s = wk.s, pc = wk.pc, b = wk.b;
      const int kvh = pc / HC;
      const int hq0 = kvh * G + (pc % HC) * GT;
      const int L = wk.L;

      float m_mine = -CUDART_INF_F;
      float l_mine = 0.f;
      float2 acc[GT][C::DPV / 2];
#pragma unroll
      for (int h = 0; h < GT; ++h)
#pragma unroll
        for (int i = 0; i < C::DPV / 2; ++i) acc[h][i] = make_float2(0.f, 0.f);

      // this warp's first tile of the segment (warps >= ncw take none)
      long long jj = warp < a.ncw ? j + ((warp - int(uint32_t(j) % uint32_t(a.ncw))) + a.ncw) % a.ncw : j + n;
      const long long jj0 = jj;
      if (jj < j + n) {
        // q slice of this lane, pre-scaled so scores come out in log2 units
        float2 qreg[GT][C::DPL / 2];
        const T *qs = static_cast<const T *>(a.q) + ((long long)s * a.Hq + hq0) * D;
#pragma unroll
        for (int h = 0; h < GT; ++h)
#pragma unroll
          for (int c = 0; c < C::CPL; ++c) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(qs + h * D + (c * C::LPT + jl) * C::EPC);
            float2 f[C::EPC / 2];
            Elem<T>::chunk_to_f2(raw, f);
#pragma unroll
            for (int i = 0; i < C::EPC / 2; ++i)
              qreg[h][c * (C::EPC / 2) + i] = make_float2(f[i].x * a.qscale, f[i].y * a.qscale);
          }

        for (; jj < j + n; jj += a.ncw) {
          const int bb = b + int(jj - j);
          const int nv = min(B, L - bb * B);
          const uint32_t ee = uint32_t(jj);  // the pair's ring entry (a CTA's count fits 32 bits)
          const int slot = int(ee % uint32_t(a.nstage));
          const char *kt = reinterpret_cast<const char *>(ring) + size_t(slot) * a.slot_stride;
          const char *vt = kt + a.tile_stride;

          // ---- wait for the pair (K and V land together), then QK
          const bool okE = wait_entry(full_bar, empty_bar, ee, a.nstage, abort_flag);
          if (!okE) {
            if (lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          __syncwarp();
          for (int t0 = 0; t0 < nv; t0 += C::TS) {
            const int t = t0 + tsub;
            const int tr = t < nv ? t : nv - 1;
            float2 a2[GT];
#pragma unroll
            for (int h = 0; h < GT; ++h) a2[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
              const uint4 raw =
                  *reinterpret_cast<const uint4 *>(kt + (size_t(tr) * D + (c * C::LPT + jl) * C::EPC) * sizeof(T));
              float2 kf[C::EPC / 2];
              Elem<T>::chunk_to_f2(raw, kf);
#pragma unroll
              for (int h = 0; h < GT; ++h)
#pragma unroll
                for (int i = 0; i < C::EPC / 2; ++i) ffma2(a2[h], qreg[h][c * (C::EPC / 2) + i], kf[i]);
            }
            float part[GT];
#pragma unroll
            for (int h = 0; h < GT; ++h) part[h] = a2[h].x + a2[h].y;
#pragma unroll
            for (int off = C::LPT / 2; off >= 1; off >>= 1)
#pragma unroll
              for (int h = 0; h < GT; ++h) part[h] += __shfl_xor_sync(kFullMask, part[h], off);
            if (t < nv && jl < GT) {
              float v = part[0];
#pragma unroll
              for (int h = 1; h < GT; ++h)
                if (jl == h) v = part[h];
              sc[t * GT + jl] = v;
            }
          }
          __syncwarp();

          // ---- online softmax over this tile (base 2)
          float mx = -CUDART_INF_F;
          for (int i = lane; i < nv * GT; i += 32) mx = fmaxf(mx, sc[i]);
#pragma unroll
          for (int off = GT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
          const float m_new = fmaxf(m_mine, mx);
          const float alpha = fast_exp2(m_mine - m_new);
          float lsum = l_mine * alpha;
          for (int i = lane; i < nv * GT; i += 32) {
            const float p = fast_exp2(sc[i] - m_new);
            sc[i] = p;
            lsum += p;
          }
          l_mine = lsum;
          m_mine = m_new;
#pragma unroll
          for (int h = 0; h < GT; ++h) {
            const float ah = __shfl_sync(kFullMask, alpha, h);
            const float2 a2 = make_float2(ah, ah);
#pragma unroll
            for (int i = 0; i < C::DPV / 2; ++i) fmul2(acc[h][i], a2);
          }
          __syncwarp();

          // ---- PV
#pragma unroll 4
          for (int t = 0; t < nv; ++t) {
            float p[GT];
            load_p<GT>(sc, t, p);
            float2 vf[C::DPV / 2];
            load_v<T, C::DPV>(vt + size_t(t) * D * sizeof(T), lane, vf);
#pragma unroll
            for (int h = 0; h < GT; ++h) {
              const float2 pp = make_float2(p[h], p[h]);
#pragma unroll
              for (int i = 0; i < C::DPV / 2; ++i) ffma2(acc[h][i], pp, vf[i]);
            }
          }
          __syncwarp();
          if (lane == 0 && okE) mbar_arrive(&empty_bar[slot]);  // the pair's slot is free again
        }
      }

      // ---- hand this warp's state for the segment to the merger warp (only
      // warps that took a tile of it)
      if (jj0 < j + n) {
        float lsum = l_mine;
#pragma unroll
        for (int off = GT; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFullMask, lsum, off);
        deposit_state(a, dep, lane, &st_full[warp][0], &st_free[warp][0], abort_flag, [&]() {
          if (lane < GT) {
            mrg[warp][lane][D] = m_mine;
            mrg[warp][lane][D + 1] = lsum;
          }
#pragma unroll
          for (int h = 0; h < GT; ++h)
#pragma unroll
            for (int i = 0; i < C::DPV / 2; ++i) {
              mrg[warp][h][lane * C::DPV + 2 * i] = acc[h][i].x;
              mrg[warp][h][lane * C::DPV + 2 * i + 1] = acc[h][i].y;
            }
        });
        ++dep;
      }
      j += n;
      wk.advance(a, n, PC);
    }
  }
}

}  // namespace pagedkv
