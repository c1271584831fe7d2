// ssm_device.cuh -- device helpers shared by the libssm kernels (sm_103a).
//
// Inline PTX for the special-function unit (ex2/lg2/rcp), packed f32x2
// arithmetic, bf16 packing, mbarriers and TMA (cp.async.bulk.tensor).
// Every spin-wait here is bounded: on timeout it records SSM device status
// bits and returns false; it never traps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// ---------------------------------------------------------------------------
// device status words (first bytes of the caller's workspace)
// ---------------------------------------------------------------------------
struct DeviceStatus {
  unsigned int flags;        // bit 0: an mbarrier wait timed out
  unsigned int where;        // kernel-specific code of the first timeout
  unsigned int pad[2];
};
constexpr unsigned int kStatusTimeout = 1u;

// A wait gives up after this much wall time (read from %globaltimer): far
// beyond any legitimate TMA completion, short enough that a broken pipeline
// ends the kernel with an error status instead of a hang.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void record_timeout(DeviceStatus* st, unsigned int where) {
  if (st) {
    if ((atomicOr(&st->flags, kStatusTimeout) & kStatusTimeout) == 0u) st->where = where;
  }
}

// ---------------------------------------------------------------------------
// special-function unit (approximate, hardware) and constants
// ---------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// division of 32-bit unsigned integers by an invariant divisor d >= 1 with one
// multiply-high, an add and two shifts (Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", PLDI 1994, the round-up method for
// N = 32: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
// q = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0) with t = mulhi(m, n))
// ---------------------------------------------------------------------------
struct FastDivU32 {
  uint32_t d, m;
  int sh1, sh2;
  __host__ __device__ static FastDivU32 make(uint32_t dv) {
    FastDivU32 f;
    f.d = dv;
    int l = 0;
    while (l < 32 && (uint64_t(1) << l) < dv) ++l;
    f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - dv)) / dv + 1);
    f.sh1 = l < 1 ? l : 1;
    f.sh2 = l > 1 ? l - 1 : 0;
    return f;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> sh1)) >> sh2;
  }
};

// ---------------------------------------------------------------------------
// packed f32x2 arithmetic (two lanes of fp32 per instruction)
// ---------------------------------------------------------------------------
struct f2 {
  float x, y;
};
__device__ __forceinline__ f2 mk2(float a, float b) { return f2{a, b}; }

__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// round both to bf16 (nearest even); lo in bits 0..15
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

// io element traits: float or bf16 (stored as uint16_t)
template <typename IO>
struct Io;
template <>
struct Io<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float load(const float* p) { return *p; }
  __device__ __forceinline__ static float ldg(const float* p) { return __ldg(p); }
  __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
};
template <>
struct Io<uint16_t> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float load(const uint16_t* p) { return bf16_to_f32(*p); }
  __device__ __forceinline__ static float ldg(const uint16_t* p) {
    return bf16_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p)));
  }
  __device__ __forceinline__ static void store(uint16_t* p, float v) { *p = f32_to_bf16(v); }
};

// ---------------------------------------------------------------------------
// exact-ish pieces for the fp32 (accurate) path
// ---------------------------------------------------------------------------
// 2^q - 1 without cancellation: Taylor series of e^x - 1 (x = q ln 2) to degree
// 4 for |q| < 1/8 (truncation below 4e-8 relative); hardware ex2 minus one
// beyond, where |2^q - 1| >= 0.083 keeps the subtraction's relative error below
// 3e-6.
constexpr float kExpm1SeriesMaxQ = 0.125f;
__device__ __forceinline__ float exp2m1_accurate(float q, float a /* = ex2(q) */) {
  // coefficients ln2^k / k!, k = 1..4
  const float c1 = 0.69314718055994531f, c2 = 0.24022650695910071f,
              c3 = 0.05550410866482158f, c4 = 0.00961812910762848f;
  float p = fmaf(c4, q, c3);
  p = fmaf(p, q, c2);
  p = fmaf(p, q, c1);
  p = p * q;
  return (fabsf(q) < kExpm1SeriesMaxQ) ? p : (a - 1.0f);
}

// |A| below this (or A == 0) sends a bf16 channel group to the accurate path: the fast
// path forms (Abar - 1) w as Abar (h + w) - w, whose absolute error grows like
// 2^-22 |B u / A|.
constexpr float kFastPathMinAbsA = 0.125f;
// A block of positions with a state update |q| = |dt A| log2(e) below this takes the
// accurate update even on the fast path: Abar (h + w) - w with Abar = ex2(q) carries an
// error of about 2^-22 |h + w| per step, which matters once it is not small against the
// exact increment (Abar - 1)(h + w) ~ q ln2 |h + w| -- a state built only from tiny steps
// (dt -> 0, the "keep the state" regime of the selection mechanism) would be lost to it.
// At 2^-15 the fast update's error stays below 2^-6.5 of each increment.
constexpr float kFastPathMinQ = 3.0517578125e-05f;  // 2^-15

// Arithmetic of a state update: the fast form Abar (h + w) - w (bf16 io), the accurate
// form for a channel whose A are all negative (2^q - 1 from exp2m1_neg, no branch), and
// the general accurate form (expm1 series near zero, the dt limit at A == 0, any sign).
constexpr int kArFast = 0, kArNeg = 1, kArGen = 2;

// softplus in log2 units: returns log2(1 + 2^x2) (= softplus(x) * log2 e for x2 = x log2 e).
// With t = 2^x2: the hardware lg2 of 1 + t while that sum keeps enough of t's bits
// (x2 >= -12: rounding 1 + t costs at most 2^-24 / t = 2^-12 relative); below, the
// series' leading term t log2(e) (log2(1 + t) = log2(e) (t - t^2/2 + ...), so its
// relative error is below t / 2 <= 2^-13) -- a vanishing step stays positive instead
// of rounding 1 + t to 1 (for x2 < -24 that would make dt exactly 0).  x itself beyond
// x2 = 20 (the rest is below 2^-20 relative).
__device__ __forceinline__ float softplus_log2_fast(float x2) {
  const float t = ex2(x2);
  const float big = lg2(1.0f + t);
  return (x2 > 20.0f) ? x2 : ((x2 < -12.0f) ? t * kLog2e : big);
}
// to about 1 ulp from the library log1pf / expf, for memory-bound kernels (decode),
// where the arithmetic costs nothing
__device__ __forceinline__ float softplus_log2_precise(float x2) {
  const float x = x2 * kLn2;
  const float sp = (x > 15.0f) ? x : log1pf(expf(x));
  return sp * kLog2e;
}

// accurate variant (fp32 io; about 3e-6 relative): max(x2, 0) + log2(1 + t) with
// t = 2^-|x2| in (0, 1]; log2(1 + t) from the hardware lg2 for t >= 1/16 (its absolute
// error, about 2^-22, is then below 3e-6 of the result) and below that from the series
// log2(e) (t - t^2/2 + t^3/3 - t^4/4) (truncation under t^4 / 5 < 3.1e-6 relative)
__device__ __forceinline__ float softplus_log2_accurate(float x2) {
  const float t = ex2(-fabsf(x2));
  const float ser = t * kLog2e * fmaf(fmaf(fmaf(-0.25f, t, 1.0f / 3.0f), t, -0.5f), t, 1.0f);
  const float l = (t < 0.0625f) ? ser : lg2(1.0f + t);
  return fmaxf(x2, 0.0f) + l;
}

// 2^q - 1 for q <= 0 without cancellation and without a branch.  Two estimates, both
// never below the true value: the degree-4 Taylor series of e^x - 1 (x = q ln 2), whose
// remainder e^xi x^5 / 120 is negative for x < 0 (accurate near zero, too large far
// from it), and the hardware 2^q minus 1 raised by 2^-22, more than that ex2's error
// (accurate away from zero).  The smaller one is the accurate one: within about 4e-8
// relative for |q| <= 1/8 and 2^-21 absolute beyond.
__device__ __forceinline__ float exp2m1_neg(float q, float a /* = ex2(q) */) {
  // coefficients ln2^k / k!, k = 1..4
  const float c1 = 0.69314718055994531f, c2 = 0.24022650695910071f,
              c3 = 0.05550410866482158f, c4 = 0.00961812910762848f;
  float p = fmaf(c4, q, c3);
  p = fmaf(p, q, c2);
  p = fmaf(p, q, c1);
  return fminf(p * q, a - 0.99999976158142089844f /* 1 - 2^-22 */);
}
// 1 - 2^q for two values q = -nq <= 0 (packed f32x2 arithmetic), from nq = -q and
// a = 2^q: the same two estimates with signs flipped, so the larger is the accurate one
__device__ __forceinline__ f2 one_minus_exp2_neg2(f2 nq, f2 a) {
  const f2 c1 = mk2(0.69314718055994531f, 0.69314718055994531f);
  const f2 c2 = mk2(-0.24022650695910071f, -0.24022650695910071f);
  const f2 c3 = mk2(0.05550410866482158f, 0.05550410866482158f);
  const f2 c4 = mk2(-0.00961812910762848f, -0.00961812910762848f);
  f2 p = fma2(c4, nq, c3);  // the series of e^x - 1 at x = -nq ln 2, in powers of nq
  p = fma2(p, nq, c2);
  p = fma2(p, nq, c1);
  p = mul2(p, nq);
  const f2 d = sub2(mk2(0.99999976158142089844f, 0.99999976158142089844f), a);
  return mk2(fmaxf(p.x, d.x), fmaxf(p.y, d.y));
}

__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// z * sigmoid(z), with sigmoid(z) = (1 + tanh(z / 2)) / 2: one hardware tanh
// (absolute error near 2^-11) instead of ex2 and rcp; for bf16 outputs
__device__ __forceinline__ float silu_fast(float z) {
  return z * fmaf(0.5f, tanh_hw(0.5f * z), 0.5f);
}
// z * sigmoid(z) to about 5e-7 relative: hardware ex2 and reciprocal (for z < -88 the
// exponential overflows to inf and the result is -0, the limit)
__device__ __forceinline__ float silu_accurate(float z) {
  return z * rcp(1.0f + ex2(-z * kLog2e));
}

// ---------------------------------------------------------------------------
// mbarrier (shared::cta) with bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// true when the phase with `parity` completed; false once `limit_ns` passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA: tiled bulk tensor copies (3-D), global <-> shared
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// load box at (c0 fastest, c1, c2) into smem, completing on `bar`
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// store smem box to global at (c0, c1, c2); out-of-range elements are not written
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until at most N committed store groups still read shared memory
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Ampere-style asynchronous 16-byte copy global -> shared (L2 only), and its
// group commit / wait (a hardware wait, not a spin loop)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(__cvta_generic_to_global(gmem_src))
               : "memory");
}
// the same copy, zero-filling the 16 bytes instead of reading when !valid
__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gmem_src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(__cvta_generic_to_global(gmem_src)), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// bulk (TMA, untiled) copy shared -> global of `bytes` (multiple of 16, both
// addresses 16-byte aligned), tracked by the bulk async-group of this thread
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   __cvta_generic_to_global(gmem_dst)),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

// 16-byte vector shared loads/stores
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ float4 lds128f(const void* p) {
  return *reinterpret_cast<const float4*>(p);
}

}  // namespace ssm
