// pa_common.cuh -- device helpers shared by the libpagedkv kernels (sm_103a):
// element conversions, packed fp32x2 FMA, mbarrier and bulk-copy (TMA) PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/pagedkv.h"

namespace pagedkv {

constexpr unsigned kFullMask = 0xffffffffu;

// ----------------------------------------------------------------- status
inline pa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t dtype_bytes(pa_dtype dt) { return dt == PA_F32 ? 4u : 2u; }

// Number of SMs of the current device (cached per device ordinal).
int device_sm_count();

// ----------------------------------------------------------------- errors
__device__ __forceinline__ void raise_error(int *err, unsigned bit) {
  if (err != nullptr) atomicOr(reinterpret_cast<unsigned *>(err), bit);
}

// Debug builds (-DPA_DEBUG) range-check every shared / global address the
// decode kernels form; an offending one is replaced by a safe one and a bit
// is raised: 1<<8 shared memory, 1<<9 tensor-copy box, 1<<10 global memory.
#ifdef PA_DEBUG
constexpr unsigned kDbgSmem = 1u << 8, kDbgTma = 1u << 9, kDbgGlobal = 1u << 10, kDbgPhase = 1u << 11;
#define PA_DBG_FIX(cond, bit, fix)  \
  do {                              \
    if (!(cond)) {                  \
      raise_error(a.err, (bit));    \
      fix;                          \
    }                               \
  } while (0)
#else
#define PA_DBG_FIX(cond, bit, fix) \
  do {                             \
  } while (0)
#endif

// ----------------------------------------------------------------- conversions
template <typename T> struct Elem;

template <> struct Elem<float> {
  // 16-byte chunk -> 4 floats as 2 float2
  static __device__ __forceinline__ void chunk_to_f2(const uint4 &c, float2 *o) {
    o[0] = make_float2(__uint_as_float(c.x), __uint_as_float(c.y));
    o[1] = make_float2(__uint_as_float(c.z), __uint_as_float(c.w));
  }
  static __device__ __forceinline__ float2 word2_to_f2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
  }
  static __device__ __forceinline__ float to_float(float x) { return x; }
  static __device__ __forceinline__ float from_float(float x) { return x; }
  // 4 consecutive outputs (16-byte aligned)
  static __device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
};

template <> struct Elem<__nv_bfloat16> {
  // bf16 is the high half of an fp32 pattern: unpack with a shift and a mask.
  static __device__ __forceinline__ float2 word_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ void chunk_to_f2(const uint4 &c, float2 *o) {
    o[0] = word_to_f2(c.x);
    o[1] = word_to_f2(c.y);
    o[2] = word_to_f2(c.z);
    o[3] = word_to_f2(c.w);
  }
  static __device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_float(float x) { return __float2bfloat16_rn(x); }
  // 4 consecutive outputs, rounded to nearest even (8-byte aligned)
  static __device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
  }
};

template <> struct Elem<__half> {
  static __device__ __forceinline__ float2 word_to_f2(uint32_t w) {
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = w;
    return __half22float2(h);
  }
  static __device__ __forceinline__ void chunk_to_f2(const uint4 &c, float2 *o) {
    o[0] = word_to_f2(c.x);
    o[1] = word_to_f2(c.y);
    o[2] = word_to_f2(c.z);
    o[3] = word_to_f2(c.w);
  }
  static __device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_float(float x) { return __float2half_rn(x); }
  // 4 consecutive outputs, rounded to nearest even (8-byte aligned)
  static __device__ __forceinline__ void store4(__half *p, float4 v) {
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
  }
};

// ----------------------------------------------------------------- packed FMA
// d.xy += a.xy * b.xy with one fma.rn.f32x2 (two IEEE fp32 FMAs).
__device__ __forceinline__ void ffma2(float2 &d, const float2 a, const float2 b) {
  uint64_t dd, aa, bb;
  asm("mov.b64 %0, {%1, %2};" : "=l"(dd) : "f"(d.x), "f"(d.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(aa) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(bb) : "f"(b.x), "f"(b.y));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(dd) : "l"(aa), "l"(bb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(dd));
}

__device__ __forceinline__ void fmul2(float2 &d, const float2 a) {
  uint64_t dd, aa;
  asm("mov.b64 %0, {%1, %2};" : "=l"(dd) : "f"(d.x), "f"(d.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(aa) : "f"(a.x), "f"(a.y));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(dd) : "l"(aa));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(dd));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------- shared memory / mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same condition (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after kWaitLimitCycles SM cycles (>= 1.4 s at the 2.07 GHz maximum clock;
// a test build of the library may set a shorter limit with PA_WAIT_LIMIT_CYCLES),
// or at once when *abort is set; returns false then.  The limit is counted on
// the SM cycle counter, which only moves forward within a thread: the global
// nanosecond timer is re-synchronised to host time and can jump forward by
// more than a second, which would end healthy waits.
#ifndef PA_WAIT_LIMIT_CYCLES
#define PA_WAIT_LIMIT_CYCLES 3000000000LL
#endif
constexpr long long kWaitLimitCycles = PA_WAIT_LIMIT_CYCLES;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  // a phase that has already completed is seen by test_wait at a fraction of
  // try_wait's cost (measured on GB300: 22 against about 200 cycles)
  if (mbar_test_wait(bar, parity)) return true;
  const long long c0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - c0 > kWaitLimitCycles) {
#ifdef PA_DEBUG
      printf("pagedkv wait gave up: cta %d thread %d bar %u parity %u after %lld cycles\n", blockIdx.x, threadIdx.x,
             smem_addr(bar), parity, (long long)(clock64() - c0));
#endif
      return false;
    }
  }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on
// `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2-D tiled bulk copy (TMA tensor) global -> shared: box at element
// coordinates (x = innermost, y) of `map`, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled bulk copy (TMA tensor) global -> shared at element coordinates
// (x innermost, y, z).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// L2 policy for data a kernel reads once: its lines are the first to go
// when L2 needs room, so that small data read again and again (tables,
// lengths, partial records) stays.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The default L2 policy, as a value for the hinted copies below.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The two tensor copies above with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, int x, int y, int z,
                                                 uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Atomic add at GPU scope with acquire-release semantics: what this thread
// wrote before it -- and what its warp wrote before a preceding __syncwarp --
// is visible to a thread that reads the counter afterwards with acquire
// semantics, and what other threads released before their own increments is
// visible to this thread's later reads.  One such atomic replaces a full
// (sequentially consistent) fence of every lane followed by a relaxed atomic.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch.  grid_dependency_wait: block until the grids
// this one depends on have completed and their writes are visible (returns at
// once when the launch did not allow an early start).  launch_dependents:
// let a dependent grid that allows it start launching now.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- warp-level MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename T> struct Mma;

template <> struct Mma<__nv_bfloat16> {
  static constexpr bool kIsBf16 = true;
  // d += A(16x16, row) * B(16x8, col), fp32 accumulate
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  // {lo, hi} -> packed pair, round to nearest even
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};

template <> struct Mma<__half> {
  static constexpr bool kIsBf16 = false;
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = w;
    return __half22float2(h);
  }
};

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace pagedkv
