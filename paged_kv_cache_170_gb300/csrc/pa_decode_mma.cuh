// pa_decode_mma.cuh -- split-context paged decode kernel on the tensor cores
// (a4), for fp16 / bf16 caches whose block size is a multiple of 16.
//
// Same schedule as the CUDA-core kernel (pa_sched.cuh): one producer warp and
// four consumer warps per CTA, one CTA range of tiles per CTA.  Differences:
//
// * Loads.  Each K or V tile (B rows of D elements, contiguous in the pool) is
//   brought in by 2-D TMA tensor copies, one per 64-column half, with the
//   128-byte swizzle: row r's 16-byte chunk c lands at chunk c ^ (r & 7), so
//   the 8-row fragment loads below never hit the same bank twice.
//
// * QK on tensor cores, transposed: S^T = K * Q^T with one mma.m16n8k16 per
//   16 tokens x 16 dims (M = tokens, N = the <= 8 query heads sharing this kv
//   head, K = dims).  The K fragment comes from ldmatrix; the q fragment stays
//   in registers for the whole segment.  Products of two 16-bit inputs are
//   exact and summed in fp32; the fp32 score is then scaled by scale*log2(e).
//
// * Online softmax in registers: each lane holds 2 heads x 2 tokens of every
//   16-token sub-tile; row maxima come from 3 xor-shuffles.
//
// * PV on tensor cores, transposed: O^T += V^T * P^T (M = dims, N = heads,
//   K = tokens).  V^T comes from ldmatrix.trans.  The accumulator layout of S^T
//   is the transpose of the operand layout P^T needs, one 8x8 movmatrix.trans
//   per half turns one into the other.  P is fed as two 16-bit terms
//   (P = P_hi + P_lo, each rounded to the input type), so the weights carry
//   ~16 significant bits and PV stays close to an fp32 product.
#pragma once

#include "pa_mma_tile.cuh"
#include "pa_sched.cuh"

namespace pagedkv {

template <typename T, int D>
__global__ void __launch_bounds__(kDecodeThreads, kCtasPerSm)
    decode_partition_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap map_k,
                                const __grid_constant__ CUtensorMap map_v) {
  constexpr int KS = D / 16;     // k-steps of QK, m-tiles of PV
  constexpr int HALVES = D / 64; // 128-byte column halves of a row
  extern __shared__ __align__(1024) unsigned char ring_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(16) float mrg[kConsumerWarps][8][state_row(D)];
  __shared__ Plan sh_plan;
  __shared__ uint32_t issued[kMaxStages];
  __shared__ int sh_abort;
  // hand-off of a warp's state: two buffers (head slots 0-3 and 4-7 of mrg[w])
  // when GT <= 4, so a warp may run one segment ahead of the merger
  __shared__ __align__(8) uint64_t st_full[kConsumerWarps][2], st_free[kConsumerWarps][2];
  __shared__ float sh_mw[kMergeScratch];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int GT = a.GT;
  const int nbuf = GT <= 4 ? 2 : 1;  // state buffers per consumer warp in mrg
  const int HC = G / GT;
  const int PC = a.Hkv * HC;
  const int B = a.B;
  volatile int *abort_flag = &sh_abort;
  // the swizzle pattern repeats every 1024 bytes: align the ring to that
  const uint32_t raw_addr = smem_addr(ring_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  unsigned char *ring = ring_raw + pad;
  const uint32_t ring_addr = raw_addr + pad;

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
      mbar_init(&st_full[w][1], 1);
      mbar_init(&st_free[w][1], 1);
    }
    sh_abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp) {
    Plan plan;
    schedule_scan(a, PC, lane, &plan);
    if (lane == 0) {
      sh_plan = plan;
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_v)) : "memory");
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
  const uint32_t tile_bytes = uint32_t(B) * D * 2;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
#ifdef PA_TRACE
    const long long tr_t0 = clock64();
#endif
    const uint64_t kv_policy = l2_evict_first_policy();  // each K/V tile is read once per step
    produce(a, PC, HC, plan, lane, full_bar, empty_bar, issued, abort_flag,
            [&](int slot, int p, int kvh, int bb, int L, int s, int pc, bool lead) {
              (void)bb;
              (void)L;
              if (p < 0 || p >= a.num_blocks) {
                raise_error(a.err, PA_DEVERR_BLOCK_ID);
                mbar_arrive(&full_bar[slot]);  // complete the phase without data
                return;
              }
              // K and V tiles of one (block, kv head) land in one slot; the full
              // tile is copied (rows past the context are masked or zeroed later).
              // A segment's lead entries also bring the chunk's q rows, so a
              // consumer never waits on a global load when it starts a segment.
              mbar_arrive_expect_tx(&full_bar[slot], 2 * tile_bytes + (lead ? a.q_bytes : 0u));
              unsigned char *dst = ring + size_t(slot) * a.slot_stride;
              if (lead) {
                long long qoff = ((long long)s * a.Hq + kvh * G + (pc % HC) * GT) * D;
                PA_DBG_FIX(qoff >= 0 && qoff + (long long)GT * D <= (long long)a.S * a.Hq * D, kDbgGlobal, qoff = 0);
                bulk_g2s(dst + a.q_offset, static_cast<const T *>(a.q) + qoff, a.q_bytes, &full_bar[slot]);
              }
              int y = (p * a.Hkv + kvh) * B;
              PA_DBG_FIX(y >= 0 && (long long)y + B <= a.num_blocks * a.Hkv * B, kDbgTma, y = 0);
              PA_DBG_FIX(smem_addr(dst) + a.slot_stride <= ring_addr + a.nstage * a.slot_stride &&
                             (smem_addr(dst) & 1023u) == 0,
                         kDbgSmem, dst = ring);
              if (HALVES == 2 && a.nops == 1) {
                tma_load_3d_hint(dst, &map_k, 0, y, 0, &full_bar[slot], kv_policy);
                tma_load_3d_hint(dst + a.tile_stride, &map_v, 0, y, 0, &full_bar[slot], kv_policy);
              } else {
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                  tma_load_2d_hint(dst + h * B * 128, &map_k, 64 * h, y, &full_bar[slot], kv_policy);
                  tma_load_2d_hint(dst + a.tile_stride + h * B * 128, &map_v, 64 * h, y, &full_bar[slot], kv_policy);
                }
              }
            });
#ifdef PA_TRACE
    if (lane == 0 && PA_TRACE_CTA(blockIdx.x))
      printf("trace cta %d producer: cycles %lld\n", blockIdx.x, clock64() - tr_t0);
#endif
    return;
  }

  if (warp == kMergerWarp) {
    // -------------------------------------------------------------- merger
    run_merger<T, D, true>(a, plan, PC, HC, G, lane, &mrg[0][0][0], 8 * state_row(D), nbuf, &st_full[0][0],
                           &st_free[0][0], sh_mw,
                           abort_flag);
    zero_empty_rows<T>(a, D, lane, 32);
#ifdef PA_TRACE
    if (lane == 0) {
      unsigned long long t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      unsigned smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      printf("tracet %d %u %llu %llu %lld\n", blockIdx.x, smid, tr_start, t1, w1 - w0);
    }
#endif
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;      // fragment row group
  const int c4 = lane & 3;      // fragment column pair

  long long j = 0;      // tiles, in this CTA's processing order
  long long dep = 0;    // states this warp deposited for the merger
#ifdef PA_TRACE
  long long tr_c0 = clock64(), tr_wk = 0, tr_tiles = 0, tr_seg = 0, tr_nseg = 0;
#endif
  // rotated processing order (see Plan); j counts tiles in that order
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
      const int kvh = wk.pc / HC;
      const int hq0 = kvh * G + (wk.pc % HC) * GT;
      const int L = wk.L;

      // running state: heads h0 = 2*c4 and h1 = 2*c4 + 1 of this lane
      float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
      float o[KS][4];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

      // this warp's first tile of the segment (warps >= ncw take none)
      long long jj = warp < a.ncw ? j + ((warp - int(uint32_t(j) % uint32_t(a.ncw))) + a.ncw) % a.ncw : j + n;
      const long long jj0 = jj;
      if (jj < j + n) {
        // q^T fragment (B operand of QK): head g of the chunk, dims 16ks + 2*c4
        // (+1), (+8); taken from the slot of the warp's first tile (a lead entry)
        uint32_t qf[KS][2];
        for (; jj < j + n; jj += a.ncw) {
          const int bb = wk.b + int(jj - j);
          const int nv = min(B, L - bb * B);
          const int nsub = (nv + 15) >> 4;
          const uint32_t ee = uint32_t(jj);  // the pair's ring entry (a CTA's count fits 32 bits)
          const int slot = int(ee % uint32_t(a.nstage));
          const uint32_t kt = ring_addr + uint32_t(slot) * a.slot_stride;
          const uint32_t vt = kt + a.tile_stride;

          // ---- wait for the pair (K and V land together)
#ifdef PA_TRACE
          long long tr_a = clock64();
#endif
          const bool okE = wait_entry(full_bar, empty_bar, ee, a.nstage, abort_flag);
#ifdef PA_TRACE
          tr_wk += clock64() - tr_a;
          ++tr_tiles;
#endif
#ifdef PA_DEBUG
          if (okE && lane == 0 && mbar_try_wait(&full_bar[slot], ((ee / uint32_t(a.nstage)) & 1u) ^ 1u)) {
            raise_error(a.err, kDbgPhase);  // the barrier ran two phases ahead of this entry
            printf("pagedkv phase ahead: cta %d warp %d entry %lld slot %d\n", blockIdx.x, warp, ee, slot);
          }
#endif
          if (!okE) {
            if (lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
#ifdef PA_DEBUG
            if (lane == 0)
              printf("pagedkv consumer: cta %d warp %d entry %lld slot %d seg s %d pc %d b %d n %d abort %d\n",
                     blockIdx.x, warp, ee, slot, wk.s, wk.pc, wk.b, n, *abort_flag);
#endif
            *abort_flag = 1;
          }
          // Lanes leave the wait loop at different iterations: reconverge before
          // the warp-collective ldmatrix / mma.sync.aligned below.
          __syncwarp();
          if (jj == jj0) {
            const unsigned char *qs = ring + size_t(slot) * a.slot_stride + a.q_offset;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              qf[ks][0] = g < GT ? *reinterpret_cast<const uint32_t *>(qs + (g * D + 16 * ks + 2 * c4) * 2) : 0u;
              qf[ks][1] = g < GT ? *reinterpret_cast<const uint32_t *>(qs + (g * D + 16 * ks + 8 + 2 * c4) * 2) : 0u;
            }
          }

          if (nv < nsub * 16) {
            // rows past the context in the last sub-tile: make them zero so a
            // zero weight times stale data cannot produce NaN
            const int rows = nsub * 16 - nv;
            for (int i = lane; i < rows * HALVES * 8; i += 32) {
              const int r = nv + i / (HALVES * 8);
              const int hc = i % (HALVES * 8);
              size_t zo = (size_t)slot * a.slot_stride + a.tile_stride + (hc >> 3) * B * 128 + r * 128 + (hc & 7) * 16;
              PA_DBG_FIX(zo + 16 <= (size_t)a.nstage * a.slot_stride, kDbgSmem, zo = 0);
              *reinterpret_cast<uint4 *>(ring + zo) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_shared();
            __syncwarp();
          }
          mma_tile<T, D>(a, kt, vt, B, nv, qf, a.qscale, m0, m1, l0, l1, o, lane, ring_addr,
                         ring_addr + uint32_t(a.nstage) * a.slot_stride);
          __syncwarp();
          if (lane == 0 && okE) mbar_arrive(&empty_bar[slot]);  // the pair's slot is free again
        }
      }

#ifdef PA_TRACE
      const long long tr_s0 = clock64();
#endif
      // ---- this warp's state for the segment: written out directly when the
      // warp alone covered a whole (s, pc), else handed to the merger warp
      if (jj0 < j + n) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          l0 += __shfl_xor_sync(kFullMask, l0, off);
          l1 += __shfl_xor_sync(kFullMask, l1, off);
        }
        const int h0 = 2 * c4, h1 = 2 * c4 + 1;
        if (complete && __popc(participants(j, n, a.ncw)) == 1) {
          // same arithmetic as the merger's one-state combine: o * (1 / l)
          const float i0 = 1.f / l0, i1 = 1.f / l1;
          const long long row0 = (long long)wk.s * a.Hq + hq0;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            if (h0 < GT) {
              store_out1<T>(a, row0 + h0, 16 * mt + g, D, o[mt][0] * i0);
              store_out1<T>(a, row0 + h0, 16 * mt + g + 8, D, o[mt][2] * i0);
            }
            if (h1 < GT) {
              store_out1<T>(a, row0 + h1, 16 * mt + g, D, o[mt][1] * i1);
              store_out1<T>(a, row0 + h1, 16 * mt + g + 8, D, o[mt][3] * i1);
            }
          }
        } else {
          const int b = nbuf == 2 ? int(dep & 1) : 0;
          const long long use = nbuf == 2 ? (dep >> 1) : dep;
          deposit_state(a, use, lane, &st_full[warp][b], &st_free[warp][b], abort_flag, [&]() {
            float(*buf)[state_row(D)] = &mrg[warp][4 * b];
            if (g == 0) {
              if (h0 < GT) {
                buf[h0][D] = m0;
                buf[h0][D + 1] = l0;
              }
              if (h1 < GT) {
                buf[h1][D] = m1;
                buf[h1][D + 1] = l1;
              }
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              if (h0 < GT) {
                buf[h0][16 * mt + g] = o[mt][0];
                buf[h0][16 * mt + g + 8] = o[mt][2];
              }
              if (h1 < GT) {
                buf[h1][16 * mt + g] = o[mt][1];
                buf[h1][16 * mt + g + 8] = o[mt][3];
              }
            }
          });
          ++dep;
        }
      }
#ifdef PA_TRACE
      tr_seg += clock64() - tr_s0;
      ++tr_nseg;
#endif
      j += n;
      wk.advance(a, n, PC);
    }
  }
#ifdef PA_TRACE
  if (lane == 0 && PA_TRACE_CTA(blockIdx.x))
    printf("trace cta %d warp %d: tiles %lld cycles %lld waiting %lld segment-ends %lld (%lld cycles)\n",
           blockIdx.x, warp, tr_tiles, clock64() - tr_c0, tr_wk, tr_nseg, tr_seg);
#endif
}

}  // namespace pagedkv
