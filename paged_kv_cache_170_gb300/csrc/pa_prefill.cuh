// pa_prefill.cuh -- prompt (prefill) attention over the paged cache.
//
// Sequence s has n new query tokens, the last n positions of its context
// (their K/V already written into the cache); the query at position p sees
// tokens 0 .. p.  One CTA takes one (sequence, kv head, tile of 64 query
// rows); a row is (prompt position i, head hh of the kv head's group of G),
// position-major, so every row of the CTA reads the same K/V tiles.
//
// A producer warp streams the tiles 0 .. last visible block through a TMA
// ring (the decode's 3-D box with the 128-byte swizzle); the four consumer
// warps each own 16 rows and ALL consume every tile in order (exact mbarrier
// parity waits), skipping the math for tiles past their own last position.
// Per 16-token sub-tile and warp, on the tensor cores (mma.m16n8k16):
//   S = Q K^T   M = 16 rows, N = 8 tokens (2 n-tiles), K = 16 dims: the K
//               tile's rows give the B operand directly by ldmatrix;
//   causal mask (token > row position -> -inf), online softmax in base 2 with
//               fp32 state (2 rows per lane, quad shuffles for row maxima);
//   O += P V    the S accumulator of the two n-tiles is, element for element,
//               the A operand P of the next MMA (rows x 16 tokens), fed as
//               two 16-bit terms P_hi + P_lo; V^T comes by ldmatrix.trans.
// Rows of a partly filled last block past the context are zeroed in the ring
// (all consumer warps, then a named barrier) so no masked weight meets stale
// data.  Output rows are normalised by their softmax sums and rounded once.
#pragma once

#include "pa_mma_tile.cuh"
#include "pa_sched.cuh"

namespace pagedkv {

struct PrefillArgs {
  void *out;
  const void *q;
  const int32_t *tables;
  const int32_t *lens;
  const int32_t *q_start;  // [S + 1] query rows of each sequence in q / out
  int64_t num_blocks;
  int max_blocks, S, Hq, Hkv, B;
  float qscale;  // scale * log2(e)
  int *err;
  int nstage, pg, nops;
  uint32_t slot_stride, tile_stride;
};

constexpr int kPrefillRows = 64;  // query rows per CTA: 4 warps x 16
constexpr int kPrefillThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingBytesPrefill = 96 * 1024;

template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads, kCtasPerSm)
    prefill_mma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v) {
  constexpr int KS = D / 16;     // k-steps of QK
  constexpr int NT = D / 8;      // n-tiles of PV (8 dims each)
  constexpr int HALVES = D / 64;
  extern __shared__ __align__(1024) unsigned char ring_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ uint32_t issued[kMaxStages];
  __shared__ int sh_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.y, kvh = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int B = a.B;
  // tiles of later prompt positions have more to read: run them first
  const int qt = int(gridDim.x) - 1 - int(blockIdx.x);
  const int q0 = a.q_start[s];
  const int n = a.q_start[s + 1] - q0;
  const long long cap = (long long)a.max_blocks * B;
  long long Lr = a.lens[s];
  Lr = Lr < 0 ? 0 : (Lr > cap ? cap : Lr);
  const int L = int(Lr);
  if (n < 0 || n > L) {  // a prompt longer than its context: nothing sensible to compute
    if (threadIdx.x == 0 && qt == 0 && kvh == 0) raise_error(a.err, PA_DEVERR_CONTEXT);
    return;
  }
  const int rows = n * G;
  const int r0 = qt * kPrefillRows;
  if (r0 >= rows) return;
  const int pos0 = L - n;                          // position of prompt token 0
  const int p_last = pos0 + (min(rows, r0 + kPrefillRows) - 1) / G;  // last position of the CTA
  const int ntile = p_last / B + 1;                // tiles the CTA reads

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
  const uint32_t tile_bytes = uint32_t(B) * D * 2;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_v)) : "memory");
    }
    const int32_t *trow = a.tables + (long long)s * a.max_blocks;
    bool aborted = false;
    for (int base = 0; base < ntile && !aborted; base += 32) {
      const int cnt = min(32, ntile - base);
      const int pid_cur = lane < cnt ? trow[base + lane] : -1;
      for (int k = 0; k < cnt; k += a.pg) {
        const int t = k + lane;
        const int pid = __shfl_sync(kFullMask, pid_cur, t < 32 ? t : 31);
        bool fail = false;
        if (lane < a.pg && t < cnt) {
          const uint32_t me = uint32_t(base + t);
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
            const int y = (pid * a.Hkv + kvh) * B;
            if (HALVES == 2 && a.nops == 1) {
              tma_load_3d(dst, &map_k, 0, y, 0, &full_bar[slot]);
              tma_load_3d(dst + a.tile_stride, &map_v, 0, y, 0, &full_bar[slot]);
            } else {
#pragma unroll
              for (int hh = 0; hh < HALVES; ++hh) {
                tma_load_2d(dst + hh * B * 128, &map_k, 64 * hh, y, &full_bar[slot]);
                tma_load_2d(dst + a.tile_stride + hh * B * 128, &map_v, 64 * hh, y, &full_bar[slot]);
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
      }
    }
    __syncwarp();
    if (lane == 0) {  // leave only when no copy into this CTA's shared memory is in flight
      for (int slot = 0; slot < a.nstage; ++slot) {
        if (issued[slot] == 0) continue;
        int never = 0;
        mbar_wait(&full_bar[slot], (issued[slot] - 1) & 1u, &never);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c4 = lane & 3;
  const int mj = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
  const int wr0 = r0 + warp * 16;             // this warp's first row
  // the lane's two rows: g and g + 8 of the warp
  const int ra = wr0 + g, rb = wr0 + g + 8;
  const int pa = pos0 + ra / G, pb = pos0 + rb / G;  // their positions
  const bool va = ra < rows, vb = rb < rows;
  const int pw = pos0 + (min(rows, wr0 + 16) - 1) / G;  // the warp's last position
  const bool active = wr0 < rows;

  // Q as the A operand: rows g / g + 8, dims 16ks + 2c4 (+1), 16ks + 8 + 2c4 (+1)
  uint32_t qa[KS][4];
  {
    const T *qra = static_cast<const T *>(a.q) + ((long long)(q0 + ra / G) * a.Hq + kvh * G + ra % G) * D;
    const T *qrb = static_cast<const T *>(a.q) + ((long long)(q0 + rb / G) * a.Hq + kvh * G + rb % G) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = va ? *reinterpret_cast<const uint32_t *>(qra + 16 * ks + 2 * c4) : 0u;
      qa[ks][1] = vb ? *reinterpret_cast<const uint32_t *>(qrb + 16 * ks + 2 * c4) : 0u;
      qa[ks][2] = va ? *reinterpret_cast<const uint32_t *>(qra + 16 * ks + 8 + 2 * c4) : 0u;
      qa[ks][3] = vb ? *reinterpret_cast<const uint32_t *>(qrb + 16 * ks + 8 + 2 * c4) : 0u;
    }
  }
  float ma = -CUDART_INF_F, mb = -CUDART_INF_F, la = 0.f, lb = 0.f;
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  int slot = 0;
  uint32_t parity = 0;
  for (int b = 0; b < ntile; ++b) {
    bool ok = !*abort_flag;
    if (ok && !mbar_wait(&full_bar[slot], parity, abort_flag)) {
      if (lane == 0 && !*abort_flag) raise_error(a.err, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
      ok = false;
    }
    __syncwarp();
    ok = __all_sync(kFullMask, ok);
    const uint32_t kt = ring_addr + uint32_t(slot) * a.slot_stride;
    const uint32_t vt = kt + a.tile_stride;
    const int t0 = b * B;
    // sub-tiles any row of the CTA can see; rows of them past the context are zeroed
    const int nsub = (min(B, p_last + 1 - t0) + 15) >> 4;
    const int zfrom = L - t0;  // first row of this block past the context
    if (zfrom < nsub * 16) {
      if (ok) {
        const int zrows = nsub * 16 - zfrom;
        for (int i = warp * 32 + lane; i < zrows * HALVES * 8; i += kConsumerWarps * 32) {
          const int r = zfrom + i / (HALVES * 8);
          const int hc = i % (HALVES * 8);
          *reinterpret_cast<uint4 *>(ring + size_t(slot) * a.slot_stride + a.tile_stride + (hc >> 3) * B * 128 +
                                     r * 128 + (hc & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_shared();
      }
      named_barrier_sync(1, kConsumerWarps * 32);
    }
    if (ok && active && t0 <= pw) {
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        if (st >= nsub || t0 + 16 * st > pw) continue;
        // ---- S = Q K^T for tokens t0 + 16 st .. +15 (n-tile 0: +0..7, n-tile 1: +8..15)
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = st * 16 + (mj >> 1) * 8 + mr;  // matrices: (tokens 0-7 | 8-15) x (dims +0 | +8)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t bf[4];
          uint32_t ad = swz(kt, B, ks >> 2, krow, (ks & 3) * 2 + (mj & 1));
          PA_DBG_FIX(ad >= ring_addr && ad + 16 <= ring_end && (ad & 15u) == 0, kDbgSmem, ad = ring_addr);
          ldmatrix_x4(bf, ad);
          Mma<T>::run(c[0], qa[ks], bf[0], bf[1]);
          Mma<T>::run(c[1], qa[ks], bf[2], bf[3]);
        }
        // ---- causal mask, online softmax (base 2)
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int tk = t0 + 16 * st + nt * 8 + 2 * c4;
          sc[nt][0] = tk <= pa ? c[nt][0] * a.qscale : -CUDART_INF_F;
          sc[nt][1] = tk + 1 <= pa ? c[nt][1] * a.qscale : -CUDART_INF_F;
          sc[nt][2] = tk <= pb ? c[nt][2] * a.qscale : -CUDART_INF_F;
          sc[nt][3] = tk + 1 <= pb ? c[nt][3] * a.qscale : -CUDART_INF_F;
        }
        float xa = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float xb = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        xa = fmaxf(xa, __shfl_xor_sync(kFullMask, xa, 1));
        xa = fmaxf(xa, __shfl_xor_sync(kFullMask, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(kFullMask, xb, 1));
        xb = fmaxf(xb, __shfl_xor_sync(kFullMask, xb, 2));
        const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
        // a row that has seen nothing yet keeps max -inf: its weights stay 0
        const float aa = na == -CUDART_INF_F ? 1.f : fast_exp2(ma - na);
        const float ab = nb == -CUDART_INF_F ? 1.f : fast_exp2(mb - nb);
        ma = na;
        mb = nb;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sc[nt][0] = na == -CUDART_INF_F ? 0.f : fast_exp2(sc[nt][0] - na);
          sc[nt][1] = na == -CUDART_INF_F ? 0.f : fast_exp2(sc[nt][1] - na);
          sc[nt][2] = nb == -CUDART_INF_F ? 0.f : fast_exp2(sc[nt][2] - nb);
          sc[nt][3] = nb == -CUDART_INF_F ? 0.f : fast_exp2(sc[nt][3] - nb);
        }
        la = la * aa + sc[0][0] + sc[0][1] + sc[1][0] + sc[1][1];
        lb = lb * ab + sc[0][2] + sc[0][3] + sc[1][2] + sc[1][3];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[nt][0] *= aa;
          o[nt][1] *= aa;
          o[nt][2] *= ab;
          o[nt][3] *= ab;
        }
        // ---- O += P V: the accumulators are the A operand, as P_hi + P_lo
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          ph[2 * nt + 0] = Mma<T>::pack(sc[nt][0], sc[nt][1]);  // row g, tokens 8nt + 2c4 (+1)
          ph[2 * nt + 1] = Mma<T>::pack(sc[nt][2], sc[nt][3]);  // row g + 8
          const float2 f0 = Mma<T>::unpack(ph[2 * nt + 0]), f1 = Mma<T>::unpack(ph[2 * nt + 1]);
          pl[2 * nt + 0] = Mma<T>::pack(sc[nt][0] - f0.x, sc[nt][1] - f0.y);
          pl[2 * nt + 1] = Mma<T>::pack(sc[nt][2] - f1.x, sc[nt][3] - f1.y);
        }
        // A fragment order: (row g, k 0-7), (row g+8, k 0-7), (row g, k 8-15), (row g+8, k 8-15)
        const uint32_t ah[4] = {ph[0], ph[1], ph[2], ph[3]};
        const uint32_t al[4] = {pl[0], pl[1], pl[2], pl[3]};
        const int vrow = st * 16 + (mj & 1) * 8 + mr;  // matrices: (tokens 0-7 | 8-15) x (dims +0 | +8)
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t bv[4];
          const int chunk = 2 * np + (mj >> 1);  // 16-byte chunk of dims 16np (+8)
          uint32_t ad = swz(vt, B, chunk >> 3, vrow, chunk & 7);
          PA_DBG_FIX(ad >= ring_addr && ad + 16 <= ring_end && (ad & 15u) == 0, kDbgSmem, ad = ring_addr);
          ldmatrix_x4_trans(bv, ad);
          Mma<T>::run(o[2 * np], ah, bv[0], bv[1]);
          Mma<T>::run(o[2 * np], al, bv[0], bv[1]);
          Mma<T>::run(o[2 * np + 1], ah, bv[2], bv[3]);
          Mma<T>::run(o[2 * np + 1], al, bv[2], bv[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
    if (++slot == a.nstage) {
      slot = 0;
      parity ^= 1u;
    }
  }

  // ---- normalise and store: o[nt] = (row g, dims 8nt + 2c4 (+1)), (row g + 8, same)
  if (!active || *abort_flag) return;
  la += __shfl_xor_sync(kFullMask, la, 1);
  la += __shfl_xor_sync(kFullMask, la, 2);
  lb += __shfl_xor_sync(kFullMask, lb, 1);
  lb += __shfl_xor_sync(kFullMask, lb, 2);
  const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
  T *oa = static_cast<T *>(a.out) + ((long long)(q0 + ra / G) * a.Hq + kvh * G + ra % G) * D;
  T *ob = static_cast<T *>(a.out) + ((long long)(q0 + rb / G) * a.Hq + kvh * G + rb % G) * D;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (va) *reinterpret_cast<uint32_t *>(oa + 8 * nt + 2 * c4) = Mma<T>::pack(o[nt][0] * ia, o[nt][1] * ia);
    if (vb) *reinterpret_cast<uint32_t *>(ob + 8 * nt + 2 * c4) = Mma<T>::pack(o[nt][2] * ib, o[nt][3] * ib);
  }
}

}  // namespace pagedkv
