// state_update.cuh -- single-token recurrent state update (decode).
//
// One step of the recurrence for every (batch, dim) channel, h updated in place
// (Mamba_Model_Report.md, section 6: ssm_step h = deltaA * h + BX,
// y = h C + D x; here with the zero-order-hold input term of the velog review,
// section 2 "Discretization").  The step moves the fp32 state twice (read and
// write, 2 * 4 * N bytes per channel) against a few bytes of token inputs, so it
// is bound by memory.  One lane owns one channel and all N of its states and
// evaluates the per-channel scalars (softplus, D skip, gate) once; each warp
// moves its 32 channels' states (32 * 4 * N contiguous bytes) between global and
// shared memory with coalesced asynchronous copies in and one bulk (TMA) copy
// out.  The arithmetic uses the accurate ZOH form (expm1 series near zero),
// which costs little at this arithmetic intensity.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

struct UpdateParams {
  int64_t batch;
  int64_t b0;        // first batch row of this launch
  int dim;
  int softplus;
  float* h;          // [batch, dim, N]
  const float* A;    // [dim, N]
  const float* D;
  const float* bias;
  const void* u;     // [batch, dim]
  const void* delta;
  const void* z;
  const void* B;     // [batch, N]
  const void* C;
  void* y;           // [batch, dim]
};

template <typename IO, int N_, bool GATE_, bool VEC_, bool EULER_ = false>
struct UpdCfg {
  static constexpr int N = N_;
  static constexpr bool GATE = GATE_;
  static constexpr bool EULER = EULER_;  // input term dt * B instead of the ZOH form
  static constexpr bool VEC = VEC_;  // h, A 16-byte aligned; B, C rows 4-element aligned
  static constexpr int THREADS = 256;
};

// 4 io values of a B or C row into fp32 registers
template <typename IO, bool VEC>
__device__ __forceinline__ void load4(const IO* p, float* out) {
  if constexpr (VEC && sizeof(IO) == 2) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    out[0] = bf16lo(w.x);
    out[1] = bf16hi(w.x);
    out[2] = bf16lo(w.y);
    out[3] = bf16hi(w.y);
  } else if constexpr (VEC) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = w.x;
    out[1] = w.y;
    out[2] = w.z;
    out[3] = w.w;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = Io<IO>::ldg(p + k);
  }
}

// One channel's step for the lane that owns it.  `hs` points at the channel's N
// states (in shared memory when staged, else in global memory); granule k of the
// lane's registers holds states 4*((k + rot) % G) .. +3, so lanes that start
// at different granules spread their 16-byte accesses over all bank groups.
// The loads that do not depend on h (the channel's A row and token inputs) are
// issued first; `wait` then waits for the staged states, so the two memory
// latencies overlap instead of adding up.
template <typename IO, typename Cfg, typename Wait>
__device__ __forceinline__ void update_channel(const UpdateParams& p, int64_t b, int d, float* hs,
                                               int rot, Wait wait) {
  constexpr int N = Cfg::N, G = N / 4;
  const int64_t ch = b * p.dim + d;
  const float* __restrict__ Ap = p.A + static_cast<int64_t>(d) * N;
  const IO* __restrict__ Bp = static_cast<const IO*>(p.B) + b * N;
  const IO* __restrict__ Cp = static_cast<const IO*>(p.C) + b * N;

  float hv[N], Av[N];
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = ((k + rot) & (G - 1)) * 4;
    if constexpr (Cfg::VEC) {
      const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ap + g));
      Av[4 * k] = a4.x; Av[4 * k + 1] = a4.y; Av[4 * k + 2] = a4.z; Av[4 * k + 3] = a4.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) Av[4 * k + i] = __ldg(Ap + g + i);
    }
  }
  const float uv = Io<IO>::ldg(static_cast<const IO*>(p.u) + ch);
  const float dv = Io<IO>::ldg(static_cast<const IO*>(p.delta) + ch);
  const float zv = Cfg::GATE ? Io<IO>::ldg(static_cast<const IO*>(p.z) + ch) : 0.0f;
  wait();
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = ((k + rot) & (G - 1)) * 4;
    if constexpr (Cfg::VEC) {
      const float4 h4 = *reinterpret_cast<const float4*>(hs + g);
      hv[4 * k] = h4.x; hv[4 * k + 1] = h4.y; hv[4 * k + 2] = h4.z; hv[4 * k + 3] = h4.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) hv[4 * k + i] = hs[g + i];
    }
  }
  const float x2 = fmaf(dv, kLog2e, p.bias ? __ldg(p.bias + d) * kLog2e : 0.0f);
  const float s = p.softplus ? softplus_log2_precise(x2) : x2;  // dt * log2(e)

  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = ((k + rot) & (G - 1)) * 4;
    float Bv[4], Cv[4];
    load4<IO, Cfg::VEC>(Bp + g, Bv);
    load4<IO, Cfg::VEC>(Cp + g, Cv);
    if constexpr (Cfg::EULER) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a0 = Av[4 * k + i];
        const float q = s * a0;
        const float ahw = ex2(q);
        const float em1 = exp2m1_accurate(q, ahw);
        const float abar = (fabsf(q) < kExpm1SeriesMaxQ) ? 1.0f + em1 : ahw;
        const float hn = fmaf(abar, hv[4 * k + i], (s * kLn2) * (Bv[i] * uv));
        hv[4 * k + i] = hn;
        if (i & 1)
          acc1 = fmaf(Cv[i], hn, acc1);
        else
          acc0 = fmaf(Cv[i], hn, acc0);
      }
    } else {
      // h + coef (A h + B u) = Abar h + coef B u with coef = (Abar - 1) / A = s f(q),
      // f(q) = (2^q - 1) / q: near zero the Taylor series of 2^q - 1 (coefficients
      // ln2^k / k!) without its last factor q, so that f(0) = ln 2 gives coef = dt at
      // A == 0 (where the bracket is B u); beyond, (Abar - 1) / q with the hardware
      // reciprocal.  States in packed f32x2 pairs (even, odd), which are also the two
      // partial sums of the contraction.
      const f2 s2 = mk2(s, s), u2 = mk2(uv, uv);
      f2 acc2 = mk2(acc0, acc1);
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const f2 a2 = mk2(Av[4 * k + i], Av[4 * k + i + 1]);
        const f2 q = mul2(s2, a2);
        const f2 ahw = mk2(ex2(q.x), ex2(q.y));
        const f2 fser = fma2(fma2(fma2(mk2(0.00961812910762848f, 0.00961812910762848f), q,
                                       mk2(0.05550410866482158f, 0.05550410866482158f)),
                                  q, mk2(0.24022650695910071f, 0.24022650695910071f)),
                             q, mk2(0.69314718055994531f, 0.69314718055994531f));
        const f2 fbig = mul2(sub2(ahw, mk2(1.0f, 1.0f)), mk2(rcp(q.x), rcp(q.y)));
        const f2 f = mk2((fabsf(q.x) < kExpm1SeriesMaxQ) ? fser.x : fbig.x,
                         (fabsf(q.y) < kExpm1SeriesMaxQ) ? fser.y : fbig.y);
        const f2 hh = mk2(hv[4 * k + i], hv[4 * k + i + 1]);
        const f2 hn = fma2(mul2(s2, f), fma2(a2, hh, mul2(mk2(Bv[i], Bv[i + 1]), u2)), hh);
        hv[4 * k + i] = hn.x;
        hv[4 * k + i + 1] = hn.y;
        acc2 = fma2(mk2(Cv[i], Cv[i + 1]), hn, acc2);
      }
      acc0 = acc2.x;
      acc1 = acc2.y;
    }
  }
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = ((k + rot) & (G - 1)) * 4;
    if constexpr (Cfg::VEC) {
      *reinterpret_cast<float4*>(hs + g) =
          make_float4(hv[4 * k], hv[4 * k + 1], hv[4 * k + 2], hv[4 * k + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) hs[g + i] = hv[4 * k + i];
    }
  }
  float yv = fmaf(p.D ? __ldg(p.D + d) : 0.0f, uv, acc0 + acc1);
  // the gate only scales y, which a bf16 output rounds to 2^-9 anyway: hardware
  // ex2 / rcp suffice there; fp32 outputs take the library expf and division
  if constexpr (Cfg::GATE) yv *= (sizeof(IO) == 2) ? silu_fast(zv) : silu_accurate(zv);
  Io<IO>::store(static_cast<IO*>(p.y) + ch, yv);
}

// Aligned path (VEC): each warp stages its 32 channels' states (32 * 4 * N
// contiguous bytes) through shared memory: coalesced 16-byte asynchronous copies
// in, one lane per channel for the arithmetic, one bulk (TMA) store out.  A warp
// whose 32 channels run past the end of the row, and the unaligned path, read and
// write h directly.
// Five CTAs of 256 threads per SM (at most 51 registers a thread): more warps with
// their states in flight (measured on B300, the 256 x 5120 x 16 decode step in a
// graph: 4 CTAs 35.0 us, 5 CTAs 33.6 us, 6 CTAs 36.6 us with register spills).
template <typename IO, typename Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 5) state_update_kernel(const UpdateParams p) {
  constexpr int N = Cfg::N, G = N / 4;
  // Launched with programmatic stream serialisation, a step's CTAs may be
  // scheduled while the previous kernel on the stream is finishing: wait for it
  // (and its writes) before touching any input, then let the next step do the same.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // grid: x over channel blocks of one batch row, y over batch rows b0 + y
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = p.b0 + blockIdx.y;
  const int d0 = blockIdx.x * Cfg::THREADS + warp * 32;
  const int d = d0 + lane;
  if constexpr (Cfg::VEC) {
    __shared__ __align__(16) float stage[Cfg::THREADS / 32][32 * N];
    float* ws = stage[warp];
    if (d0 + 32 <= p.dim) {
      float* hrow = p.h + (b * p.dim + d0) * N;
#pragma unroll
      for (int k = 0; k < G; ++k) cp_async16(ws + (k * 32 + lane) * 4, hrow + (k * 32 + lane) * 4);
      cp_async_commit();
      // start granule per lane: 8 consecutive lanes cover all 8 bank groups
      const int rot = (lane >> (G == 4 ? 1 : G == 2 ? 2 : 3)) & (G - 1);
      update_channel<IO, Cfg>(p, b, d, ws + lane * N, rot, [] {
        cp_async_wait_all();
        __syncwarp();
      });
      fence_proxy_async_smem();  // the lanes' stores -> visible to the bulk copy
      __syncwarp();
      if (lane == 0) {
        bulk_store(hrow, ws, 32 * N * 4);
        tma_store_commit();
        tma_store_wait_read<0>();  // the copy has read the staging buffer
      }
      return;
    }
  }
  if (d < p.dim) update_channel<IO, Cfg>(p, b, d, p.h + (b * p.dim + d) * N, 0, [] {});
}

}  // namespace ssm
