// pa_decode_shared.cuh -- two of the three kernels of the shared-block decode
// (the third, for the dense groups, is prefill_tc_kernel's groups mode in
// pa_prefill.cuh: shared groups of 32 or more query rows per kv head, 128
// rows against a chunk of the run per CTA, on the tensor cores):
//
// decode_shared_mma_kernel (step 1): every other group's blocks against the
//   query rows of all its members: the smaller shared groups' runs of full
//   blocks, and each sequence's own group (its private blocks, the last one
//   partly filled).  A CTA walks its pieces (plan: c_poff, c_opoff) in
//   order; one producer warp streams each piece's K and V tiles into a ring
//   by TMA.  The four consumer warps take the unit's pass of up to 32 query
//   rows (row = member * G + head) as wr row-warps of 8 rows times 4 / wr
//   tile-lanes: with 32 rows all four warps work on every tile, so a tile
//   read once serves 32 rows of up to 32 sequences; with 8 rows (every own
//   group) each warp takes every fourth tile (tile t of piece p to lane
//   (t + p) mod 4).  Each tile-lane that got a tile leaves one partial state
//   (acc, m, l) per row of its pass in `records`, at record row
//   tl * wr * 8 + row of the piece.  Every consumer waits for every entry in
//   order, so the ring's mbarrier parity waits are exact (no warp can lag a
//   full ring behind another).  Launched early beside the tensor-core
//   kernel when there is one, it waits for that grid before it exits.
//
// merge_shared_kernel (step 2): per output row (s, h), the partial states the
//   plan lists for it (r_off, r_rec): every tile-lane state of every piece of
//   every group s belongs to,
//     M = max_i m_i;  out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
#pragma once

#include "pa_mma_tile.cuh"
#include "pa_sched.cuh"
#include "pa_share_plan.h"

namespace pagedkv {

struct SharedArgs {
  const void *q;
  const int32_t *tables;
  const int32_t *lens;  // context lengths (the own groups' last blocks may be partly filled)
  const int32_t *plan;  // device copy of the plan
  SharePlanHeader h;    // its header
  int64_t num_blocks;
  int max_blocks, S, Hq, Hkv, B;
  float qscale;      // scale * log2(e)
  float *records;    // [num_pieces][kSharePassRows][state_row(D)]
  int *err;
  int nstage, pg, nops;
  uint32_t slot_stride, tile_stride;
};

constexpr int kSharedThreads = (kConsumerWarps + 1) * 32;

constexpr int kRingBytesShared = 88 * 1024;  // ring of K + V tile pairs

// A piece's descriptor (three 16-byte loads through the read-only path).
__device__ __forceinline__ PieceDesc load_piece(const int32_t *plan, int desc_off, int p) {
  const int4 *d = reinterpret_cast<const int4 *>(plan + desc_off) + 3 * p;
  const int4 x = __ldg(d), y = __ldg(d + 1), z = __ldg(d + 2);
  PieceDesc r;
  r.unit = x.x; r.t0 = x.y; r.t1 = x.z; r.group = x.w;
  r.kvh = y.x; r.pass = y.y; r.leader = y.z; r.blk0 = y.w;
  r.moff = z.x; r.rows = z.y; r.prows = z.z; r.own = z.w;
  return r;
}

// The CTA's pieces in the order it works them: those of own units (short,
// their start latency overlaps the ring filling up), then those of shared units.
struct PieceList {
  int o0, no, s0, n;
  __device__ __forceinline__ int at(int k) const { return k < no ? o0 + k : s0 + (k - no); }
};

__device__ __forceinline__ PieceList cta_pieces(const int32_t *P, const SharePlanHeader &h) {
  PieceList l;
  l.o0 = P[h.c_opoff + blockIdx.x];
  l.no = P[h.c_opoff + blockIdx.x + 1] - l.o0;
  l.s0 = P[h.c_poff + blockIdx.x];
  l.n = l.no + P[h.c_poff + blockIdx.x + 1] - l.s0;
  return l;
}

template <typename T, int D>
__global__ void __launch_bounds__(kSharedThreads, kCtasPerSm)
    decode_shared_mma_kernel(const SharedArgs a, const __grid_constant__ CUtensorMap map_k,
                             const __grid_constant__ CUtensorMap map_v) {
  constexpr int KS = D / 16;
  constexpr int HALVES = D / 64;
  constexpr int R = state_row(D);
  extern __shared__ __align__(1024) unsigned char ring_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ uint32_t issued[kMaxStages];
  __shared__ int sh_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#ifdef PA_TRACE
  unsigned long long tg0, tg_first = 0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tg0));
#endif
  const int32_t *P = a.plan;
  const SharePlanHeader &h = a.h;
  const int Gq = h.group_size;
  const int B = a.B;
  volatile int *abort_flag = &sh_abort;
  const uint32_t raw_addr = smem_addr(ring_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  unsigned char *ring = ring_raw + pad;
  const uint32_t ring_addr = raw_addr + pad;
  const uint32_t ring_end = ring_addr + uint32_t(a.nstage) * a.slot_stride;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nstage; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
      issued[i] = 0;
    }
    sh_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const PieceList pl = cta_pieces(P, h);
  const uint32_t tile_bytes = uint32_t(B) * D * 2;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_v)) : "memory");
    }
    uint32_t e = 0;
    bool aborted = false;
    // a group read in one pass reads each of its tiles once per step: let
    // those lines go first from L2; a group of several passes reads its tiles
    // once per pass, so they keep the default policy
    const uint64_t pol_once = l2_evict_first_policy(), pol_again = l2_evict_normal_policy();
    PieceDesc nxt = pl.n > 0 ? load_piece(P, h.p_desc, pl.at(0)) : PieceDesc{};
    for (int k = 0; k < pl.n && !aborted; ++k) {
      const PieceDesc d = nxt;
      if (k + 1 < pl.n) nxt = load_piece(P, h.p_desc, pl.at(k + 1));  // the next piece's, while this one streams
      const uint64_t pol = d.rows <= d.prows ? pol_once : pol_again;
      const int32_t *trow = a.tables + (long long)d.leader * a.max_blocks + d.blk0;
      const int n = d.t1 - d.t0;
      for (int base = 0; base < n && !aborted; base += 32) {
        const int cnt = min(32, n - base);
        const int pid_cur = lane < cnt ? trow[base + lane] : -1;
        for (int kk = 0; kk < cnt; kk += a.pg) {
          const int t = kk + lane;
          const int pid = __shfl_sync(kFullMask, pid_cur, t < 32 ? t : 31);
          bool fail = false;
          if (lane < a.pg && t < cnt) {
            const uint32_t me = e + uint32_t(lane);
            const int slot = int(me % uint32_t(a.nstage));
            const uint32_t use = me / uint32_t(a.nstage);
            if (*abort_flag || (use > 0 && !mbar_wait(&empty_bar[slot], (use - 1) & 1u, abort_flag))) {
              fail = true;
            } else if (pid < 0 || pid >= a.num_blocks) {
              raise_error(a.err, PA_DEVERR_BLOCK_ID);
              mbar_arrive(&full_bar[slot]);  // complete the phase without data
              issued[slot] = use + 1;
            } else {
              mbar_arrive_expect_tx(&full_bar[slot], 2 * tile_bytes);
              unsigned char *dst = ring + size_t(slot) * a.slot_stride;
              const int y = (pid * a.Hkv + d.kvh) * B;
              if (HALVES == 2 && a.nops == 1) {
                tma_load_3d_hint(dst, &map_k, 0, y, 0, &full_bar[slot], pol);
                tma_load_3d_hint(dst + a.tile_stride, &map_v, 0, y, 0, &full_bar[slot], pol);
              } else {
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh) {
                  tma_load_2d_hint(dst + hh * B * 128, &map_k, 64 * hh, y, &full_bar[slot], pol);
                  tma_load_2d_hint(dst + a.tile_stride + hh * B * 128, &map_v, 64 * hh, y, &full_bar[slot], pol);
                }
              }
              issued[slot] = use + 1;
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
          e += uint32_t(min(a.pg, cnt - kk));
        }
      }
    }
    // leave only when no copy into this CTA's shared memory is in flight
    __syncwarp();
    if (lane == 0) {
      for (int slot = 0; slot < a.nstage; ++slot) {
        if (issued[slot] == 0) continue;
        int never = 0;
        mbar_wait(&full_bar[slot], (issued[slot] - 1) & 1u, &never);
      }
    }
    // launched early beside the tensor-core groups' kernel (whose records
    // this kernel never reads): never complete before it, so that the merge
    // after this kernel sees its records too (a no-op on a plain launch)
    grid_dependency_wait();
    return;
  }

  // -------------------------------------------------------------- consumers
  // All four consumer warps walk every entry in the same order and meet at
  // the same named barriers (id 1, 128 threads); after a timeout they keep
  // walking without waiting or computing, so no warp is left at a barrier.
  const int g8 = lane >> 2;  // fragment row group: this lane's query column
  const int c4 = lane & 3;
  int slot = 0;         // ring slot of the next entry
  uint32_t parity = 0;  // its use's parity; entries are consumed in order, one by one
#ifdef PA_TRACE
  long long tr_c0 = clock64(), tr_setup = 0, tr_wait = 0, tr_math = 0, tr_end = 0, tr_tiles = 0;
#endif
  PieceDesc nxt = pl.n > 0 ? load_piece(P, h.p_desc, pl.at(0)) : PieceDesc{};
  for (int k = 0; k < pl.n; ++k) {
#ifdef PA_TRACE
    const long long tr_p0 = clock64();
#endif
    const PieceDesc d = nxt;
    const int p = pl.at(k);
    if (k + 1 < pl.n) nxt = load_piece(P, h.p_desc, pl.at(k + 1));  // the next piece's, while this one runs
    const int n = d.t1 - d.t0;
    // wr row-warps cover the pass's rows (8 each); the 4 / wr tile-lanes take
    // every (4 / wr)-th tile, so a pass of few rows still keeps all warps busy
    const int prow = d.pass * d.prows;
    const int wr = share_row_warps(min(d.prows, d.rows - prow));
    const int rw = warp % wr, tl = warp / wr, nl = kConsumerWarps / wr;
    const int rb = prow + rw * 8;  // this warp's first row
    const int myrows = tl < nl ? max(0, min(8, d.rows - rb)) : 0;
    // an own group's last block may be partly filled: its tokens end at L
    // (its pass has at most 8 rows, so one warp computes each of its tiles)
    int L = 0;
    if (d.own) {
      const int cap = a.max_blocks * B;
      L = a.lens[d.leader];
      L = L < 0 ? 0 : (L > cap ? cap : L);
    }

    uint32_t qf[KS][2];
    if (g8 < myrows) {
      const int r = rb + g8;
      const int seq = d.own ? d.leader : P[h.g_members + d.moff + r / Gq];
      const T *qrow = static_cast<const T *>(a.q) + ((long long)seq * a.Hq + d.kvh * Gq + r % Gq) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * c4);
        qf[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * c4);
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) qf[ks][0] = qf[ks][1] = 0u;
    }
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

#ifdef PA_TRACE
    qf[0][0] = __shfl_sync(kFullMask, qf[0][0], lane);  // wait for the q loads
    tr_setup += clock64() - tr_p0;
#endif
    for (int t = 0; t < n; ++t) {
#ifdef PA_TRACE
      const long long tr_w0 = clock64();
#endif
      bool ok = !*abort_flag;
      if (ok && !mbar_wait(&full_bar[slot], parity, abort_flag)) {
        if (lane == 0 && !*abort_flag) raise_error(a.err, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
      }
      __syncwarp();
      ok = __all_sync(kFullMask, ok);
#ifdef PA_TRACE
      if (tg_first == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tg_first));
#endif
      const uint32_t kt = ring_addr + uint32_t(slot) * a.slot_stride;
#ifdef PA_TRACE
      const long long tr_m0 = clock64();
      tr_wait += tr_m0 - tr_w0;
#endif
      if (ok && myrows > 0 && (t + p) % nl == tl) {
        // shared blocks are full; an own group's last block holds L - blk * B tokens
        const int nv = d.own ? min(B, L - (d.blk0 + t) * B) : B;
        const int padded = ((nv + 15) >> 4) * 16;
        if (nv < padded) {
          // rows past the context in the last 16-row group: zero them so a zero
          // weight never meets stale data (then order these writes before the
          // slot's next bulk copy)
          for (int i = lane; i < (padded - nv) * HALVES * 8; i += 32) {
            const int r = nv + i / (HALVES * 8), hc = i % (HALVES * 8);
            const uint32_t zo = uint32_t(slot) * a.slot_stride + a.tile_stride + uint32_t((hc >> 3) * B * 128 +
                                                                                       r * 128 + (hc & 7) * 16);
            *reinterpret_cast<uint4 *>(ring + zo) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_shared();
          __syncwarp();
        }
        mma_tile<T, D>(a, kt, kt + a.tile_stride, B, nv, qf, a.qscale, m0, m1, l0, l1, o, lane, ring_addr,
                       ring_end);
#ifdef PA_TRACE
        o[0][0] = __shfl_sync(kFullMask, o[0][0], lane);
        tr_math += clock64() - tr_m0;
        ++tr_tiles;
#endif
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
      if (++slot == a.nstage) {
        slot = 0;
        parity ^= 1u;
      }
    }

#ifdef PA_TRACE
    const long long tr_e0 = clock64();
#endif
    // ---- the piece's partial state per row (acc, m, l), straight to the
    // record rows of this tile-lane (no wait for the other warps)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFullMask, l0, off);
      l1 += __shfl_xor_sync(kFullMask, l1, off);
    }
    const int h0 = 2 * c4, h1 = 2 * c4 + 1;
    if (myrows > 0 && share_lane_has_tile(p, n, tl, nl)) {
      float *dst = a.records + ((long long)p * kSharePassRows + tl * wr * 8 + rw * 8) * R;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        if (h0 < myrows) {
          dst[h0 * R + 16 * mt + g8] = o[mt][0];
          dst[h0 * R + 16 * mt + g8 + 8] = o[mt][2];
        }
        if (h1 < myrows) {
          dst[h1 * R + 16 * mt + g8] = o[mt][1];
          dst[h1 * R + 16 * mt + g8 + 8] = o[mt][3];
        }
      }
      if (g8 == 0) {
        if (h0 < myrows) {
          dst[h0 * R + D] = m0;
          dst[h0 * R + D + 1] = l0;
        }
        if (h1 < myrows) {
          dst[h1 * R + D] = m1;
          dst[h1 * R + D + 1] = l1;
        }
      }
    }
#ifdef PA_TRACE
    tr_end += clock64() - tr_e0;
#endif
  }
#ifdef PA_TRACE
  if (lane == 0 && warp == 0) {  // every CTA: start, first tile, end of consumer warp 0
    unsigned long long tg1;
    unsigned sm;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tg1));
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    printf("traces1 %d %u %llu %llu %llu %d\n", blockIdx.x, sm, tg0, tg_first, tg1, pl.n);
  }
  if (lane == 0 && PA_TRACE_CTA(blockIdx.x))
    printf("trace shared cta %d warp %d: pieces %d tiles %lld cycles %lld setup %lld wait %lld math %lld end %lld\n",
           blockIdx.x, warp, pl.n, tr_tiles, clock64() - tr_c0, tr_setup, tr_wait, tr_math, tr_end);
#endif
}

struct MergeArgs {
  void *out;             // [S][Hq][D], element type T
  const float *records;  // step 1's partial states
  const int32_t *plan;
  SharePlanHeader h;
  int S, Hq;
};

constexpr int kMergeWarps = 8;

// One warp per output row; lane i owns dims 4i .. 4i+3 (D = 128) or
// 2i .. 2i+1 (D = 64).  The row's records are listed in the plan (r_off,
// r_rec); their (m, l) come in one batch of loads, one record per lane, so
// the weights
//     w_j = 2^(m_j - M) / sum_j 2^(m_j - M) l_j,   M = max_j m_j,
// are formed before any row is read; the rows then load eight at a time.  A
// row with more than 32 records takes the weights in batches of 32, after a
// first pass for M.  A row with no record at all (empty sequence) is zero.
template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_shared_kernel(const MergeArgs a) {
  constexpr int R = state_row(D);
  constexpr int V = D / 32;  // dims per lane
  const long long row = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
#ifdef PA_TRACE
  unsigned long long tm0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tm0));
#endif
  if (row >= (long long)a.S * a.Hq) return;
  const int32_t *P = a.plan;
  const SharePlanHeader &h = a.h;
  const int k0 = P[h.r_off + row], k1 = P[h.r_off + row + 1];

  float M = -CUDART_INF_F;
  if (k1 - k0 > 32) {  // pass 1 (long lists only): M over all records
    for (int base = k0; base < k1; base += 32) {
      const int k = base + lane;
      M = fmaxf(M, k < k1 ? __ldcg(a.records + (long long)P[h.r_rec + k] * R + D) : -CUDART_INF_F);
    }
  }
  float num[V];
#pragma unroll
  for (int v = 0; v < V; ++v) num[v] = 0.f;
  float den = 0.f;
  for (int base = k0; base < k1; base += 32) {
    // this batch's records, one per lane, and their weights
    const int k = base + lane;
    const long long rid = k < k1 ? (long long)P[h.r_rec + k] : 0;
    const float *rl = a.records + rid * R;
    const float m = k < k1 ? __ldcg(rl + D) : -CUDART_INF_F;
    const float l = k < k1 ? __ldcg(rl + D + 1) : 0.f;
    if (k1 - k0 <= 32) {
      M = m;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    }
    const float f = m > -CUDART_INF_F ? fast_exp2(m - M) : 0.f;
    float dl = f * l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dl += __shfl_xor_sync(kFullMask, dl, off);
    den += dl;
    // the rows, eight records' loads in flight at a time
    const int n = min(32, k1 - base);
    for (int j0 = 0; j0 < n; j0 += 8) {
      float x[8][V];
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + i;
        const long long rj = __shfl_sync(kFullMask, rid, j & 31);
        w[i] = j < n ? __shfl_sync(kFullMask, f, j & 31) : 0.f;
        const float *rec = a.records + rj * R + lane * V;
        if constexpr (V == 4) {
          const float4 y = j < n ? __ldcg(reinterpret_cast<const float4 *>(rec)) : make_float4(0.f, 0.f, 0.f, 0.f);
          x[i][0] = y.x;
          x[i][1] = y.y;
          x[i][2] = y.z;
          x[i][3] = y.w;
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) x[i][v] = j < n ? __ldcg(rec + v) : 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int v = 0; v < V; ++v) num[v] += w[i] * x[i][v];
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T *o = static_cast<T *>(a.out) + row * D + lane * V;
#pragma unroll
  for (int v = 0; v < V; ++v) o[v] = Elem<T>::from_float(num[v] * inv);
#ifdef PA_TRACE
  if (threadIdx.x == 0) {
    unsigned long long tm1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tm1));
    printf("tracem %d %llu %llu\n", blockIdx.x, tm0, tm1);
  }
#endif
}

}  // namespace pagedkv
