// Shared device helpers of the sm_103a library: error word, mbarriers with
// bounded waits, 1-D bulk (TMA) copies, order-preserving keys, reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "eagle.h"

namespace eagle {

// ---------------------------------------------------------------- workspace
// Every workspace starts with this 256-byte header; kernels record the first
// device-side problem in `error` / `detail`.
struct WsHeader {
  int32_t error;
  int32_t detail;
  int32_t test_flags;     // test hook (zero in normal use): kTestNoCopies
  int32_t test_wait_us;   // test hook: wait limit in microseconds (0: the default 2 s)
  int32_t pad[60];
};
// test_flags bit: the attention kernel's producers issue no copy at all, so
// every consumer wait runs out (with nothing in flight) -- how the tests make
// a bounded device wait expire.
constexpr int32_t kTestNoCopies = 1;
constexpr size_t kWsHeader = sizeof(WsHeader);
static_assert(kWsHeader == 256, "header size");

constexpr int32_t kDevTimeout = EAGLE_ERR_TIMEOUT;
constexpr int32_t kDevAssert = EAGLE_ERR_DEVICE_ASSERT;

__device__ __forceinline__ void record_error(int32_t* err, int32_t code, int32_t detail) {
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, detail);
}

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

// ------------------------------------------------------------------ timing
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// `limit_ns` of wall time and returns false (the caller records a timeout).
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                       uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}


// 1-D bulk copy global -> this CTA's shared memory; completes `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 4-byte asynchronous global -> shared copy (completes per thread).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// --------------------------------------------------------- ordering / keys
// (value desc, index asc): does (va, ia) come before (vb, ib)?
// Written with bitwise operators so that it compiles to predicates, not branches.
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return (va > vb) | ((va == vb) & (ia < ib));
}

// Monotone map of a double to uint64 (larger value -> larger key); -0 == +0.
__device__ __forceinline__ uint64_t order_key(double x) {
  uint64_t u = static_cast<uint64_t>(__double_as_longlong(x));
  if (u == (1ull << 63)) u = 0;   // -0 -> +0
  return (u >> 63) ? ~u : (u | (1ull << 63));
}

// Inverse of order_key.
__device__ __forceinline__ double key_value(uint64_t k) {
  const uint64_t u = (k >> 63) ? (k & ~(1ull << 63)) : ~k;
  return __longlong_as_double(static_cast<long long>(u));
}

// 2^x on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------- exp / log to ~1e-7 relative
// The fp64 special functions are very slow on this part; these reduce the
// argument in fp64 and evaluate the remaining small range with the fp32
// library function.
//   exp(d) = 2^n * exp(r),  n = round(d / ln 2),  r = d - n ln 2 in [-0.35, 0.35]
//   (0 below e^-708, where a probability no longer matters)
//   log(s) = e ln 2 + log(f_hi) + (f - f_hi) / f_hi,  s = f 2^e, f in [0.5, 1)
__device__ __forceinline__ double exp_d(double d) {
  if (d < -708.0) return 0.0;   // below the normal range: negligible as a probability
  if (d > 709.0) d = 709.0;
  const double n = rint(d * 1.4426950408889634);
  const double r = fma(-n, 0.6931471805599453, d);   // ln 2 to double precision
  // 2^n from its exponent bits (n in [-1022, 1023])
  const double two_n = __longlong_as_double(static_cast<long long>(static_cast<int>(n) + 1023) << 52);
  return static_cast<double>(expf(static_cast<float>(r))) * two_n;
}
__device__ __forceinline__ double log_d(double s) {
  int e;
  const double f = frexp(s, &e);
  const float fh = static_cast<float>(f);
  return e * 0.6931471805599453 + static_cast<double>(logf(fh)) +
         (f - static_cast<double>(fh)) / static_cast<double>(fh);
}

// --------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp-wide best (value desc, index asc); every lane gets the winner.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    const bool t = before(ov, oi, v, i);
    v = t ? ov : v;
    i = t ? oi : i;
  }
}

}  // namespace eagle

namespace eagle {

// ------------------------------------------------ packed fp32 pairs, 3-way max
// Two fp32 lanes in one 64-bit register (fma / add on both at once, one
// instruction each), and the three-input maximum.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Programmatic dependent launch (see pdl_attribute): let the next kernel in
// the stream launch now / wait until the previous kernel has completed and
// its memory operations are visible (no-ops without the launch attribute).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over `nthreads` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace eagle
