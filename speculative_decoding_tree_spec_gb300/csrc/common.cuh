// common.cuh -- device helpers of the verify kernels: Philox4x32-10, order keys,
// element loads, tempered weights, fixed-point masses and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "internal.h"

namespace svk {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Checked builds (compiled with -DSPEC_CHECK): an index found outside its range
// sets a bit of this translation unit's error word and is replaced by 0, so the
// access stays inside its buffer; spec_check_errors() reads and clears the words.
// Other builds compile the checks to nothing.
// ---------------------------------------------------------------------------
#ifdef SPEC_CHECK
static __device__ unsigned int g_spec_check;
#define SPEC_CHECK_INDEX(i, n, bit)                                                    \
  do {                                                                                 \
    if ((unsigned long long)(long long)(i) >= (unsigned long long)(long long)(n)) {    \
      atomicOr(&::svk::g_spec_check, 1u << (bit));                                     \
      (i) = 0;                                                                         \
    }                                                                                  \
  } while (0)
#else
#define SPEC_CHECK_INDEX(i, n, bit) \
  do {                              \
  } while (0)
#endif

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies, the key advanced
// by the golden-ratio / sqrt(3) Weyl increments between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox10(uint4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t a = 0xD2511F53u, b = 0xCD9E8D57u;
    uint32_t lo_a = a * x.x, hi_a = __umulhi(a, x.x);
    uint32_t lo_b = b * x.z, hi_b = __umulhi(b, x.z);
    x = make_uint4(hi_b ^ x.y ^ k0, lo_b, hi_a ^ x.w ^ k1, lo_a);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return x;
}

__device__ __forceinline__ uint4 philox_words(uint64_t seed, uint64_t offset, int b, int node) {
  return philox10(make_uint4((uint32_t)node, (uint32_t)b, (uint32_t)offset,
                             (uint32_t)(offset >> 32)),
                  (uint32_t)seed, (uint32_t)(seed >> 32));
}

// Uniform on (0, 1]: ((x >> 8) + 1) * 2^-24, exact in fp32 and fp64.
__device__ __forceinline__ double unit_uniform(uint32_t x) {
  return (double)((x >> 8) + 1u) * (1.0 / 16777216.0);
}

// ---------------------------------------------------------------------------
// Order keys: larger logit -> larger key; -0 is folded onto +0 first.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t u = __float_as_uint(__fadd_rn(z, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// For bf16 logits the order key's low 16 bits are constant (0 above zero, 0xffff
// below), so key >> 16 is an exact 16-bit order key; this maps it back.
__device__ __forceinline__ uint32_t key_from16(uint32_t k16) {
  return (k16 << 16) | ((k16 & 0x8000u) ? 0u : 0xffffu);
}

// ---------------------------------------------------------------------------
// Element access.  A "unit" is one 16-byte vector: 4 fp32 or 8 bf16 logits.
// ---------------------------------------------------------------------------
template <typename T> struct Elt;
template <> struct Elt<float> {
  static constexpr int kPerUnit = 4;
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static float at(const void* row, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  }
};
template <> struct Elt<uint16_t> {  // bf16 stored as raw bits
  static constexpr int kPerUnit = 8;
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  __device__ __forceinline__ static float at(const void* row, int64_t i) {
    uint32_t bits = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
    return __uint_as_float(bits << 16);
  }
};

// Load unit u of a row into f[]; the partial last unit is filled with -inf.
template <typename T>
__device__ __forceinline__ void load_unit(const void* row, int V, int u,
                                          float (&f)[Elt<T>::kPerUnit]) {
  constexpr int E = Elt<T>::kPerUnit;
  int base = u * E;
  if (base + E <= V) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + u);
    Elt<T>::unpack(v, f);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = (base + e < V) ? Elt<T>::at(row, base + e) : -CUDART_INF_F;
  }
}

// ---------------------------------------------------------------------------
// Tempered weights.  Every pass that needs the weight of a token evaluates this
// one expression, so the same logit always yields the same fp32 weight:
//   w(z) = 2^((z - m) * c),  c = log2(e) / T.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tempered_weight(float z, float m, float c) {
  return ex2_approx(__fmul_rn(__fsub_rn(z, m), c));
}

// Fixed-point mass with 42 fractional bits (weights lie in [0, 1]; sums over up to
// 2^21 tokens fit in 63 bits).  Integer-only conversion with round-half-up, so a
// sum of masses is exact and independent of summation order.
constexpr int kFixBits = 42;
__device__ __forceinline__ uint64_t to_fixed(float w) {
  uint32_t u = __float_as_uint(w);
  int e = (int)(u >> 23) - 127;
  if ((u >> 23) == 0 || e < -(kFixBits + 1)) return 0ull;
  uint64_t mant = (uint64_t)((u & 0x7fffffu) | 0x800000u);
  int sh = e - 23 + kFixBits;
  if (sh >= 0) return mant << sh;
  int s = -sh;
  return (mant + (1ull << (s - 1))) >> s;
}
__device__ __forceinline__ double fixed_to_double(uint64_t x) {
  return (double)x * (1.0 / 4398046511104.0);  // 2^-42
}

// ---------------------------------------------------------------------------
// Warp / block reductions.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Float-float (hi, lo) arithmetic: error-free two-sum in fp32.  Used instead of
// per-thread fp64, whose throughput on this part is a small fraction of fp32.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
struct FF {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    float s, e;
    two_sum(hi, x, s, e);
    lo += e;
    hi = s;
  }
  __device__ __forceinline__ void add(const FF& o) {
    float s, e;
    two_sum(hi, o.hi, s, e);
    lo += e + o.lo;
    hi = s;
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};
// Butterfly sum of a float-float value over the warp (every lane gets the total).
__device__ __forceinline__ FF warp_sum_ff(FF v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    FF t;
    t.hi = __shfl_xor_sync(kFull, v.hi, o);
    t.lo = __shfl_xor_sync(kFull, v.lo, o);
    v.add(t);
  }
  return v;
}

// 16-byte asynchronous global -> shared copies (each thread later reads only the
// bytes it copied itself, so no block barrier is needed between stages).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// mbarriers and bulk (TMA) copies.  Every wait is bounded in time: once
// `limit_ns` have passed (read from %globaltimer) it gives up and returns false,
// and the caller records a timeout and carries on without waiting again, so no
// wait -- and no barrier behind it -- can hold the GPU.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
                   smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for the phase with `parity` to complete; false once limit_ns have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 32; ++k)
      if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
// Bulk global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that signals `bar` with its byte count on completion.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Named barrier over the first `nthreads` threads of the block (barrier id 1).
__device__ __forceinline__ void named_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;\n" ::"r"(nthreads) : "memory");
}

// Kahan-compensated fp32 accumulator.
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    float y = x - c;
    float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s - (double)c; }
  __device__ __forceinline__ FF ff() const {
    FF r;
    two_sum(s, -c, r.hi, r.lo);
    return r;
  }
};

}  // namespace svk
