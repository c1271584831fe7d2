// state_update.cuh -- single-token recurrent state update (decode).
//
// One step of the recurrence for every (batch, dim) channel, h updated in place
// (Mamba_Model_Report.md, section 6: ssm_step h = deltaA * h + BX,
// y = h C + D x; here with the zero-order-hold input term of the velog review,
// section 2 "Discretization").  The step moves the fp32 state twice (read and
// write, 2 * 4 * N bytes per channel) against a few bytes of token inputs, so
// it is bound by HBM: four lanes share a channel's 16 states as one 16-byte
// vector each, a warp reads 512 contiguous bytes of h, and the contraction is
// summed with two xor-shuffles.  The arithmetic uses the accurate ZOH form
// (expm1 series near zero) since it costs nothing at this arithmetic intensity.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

struct UpdateParams {
  int64_t channels;  // batch * dim
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

template <typename IO, int N_, bool GATE_, bool VEC_>
struct UpdCfg {
  static constexpr int N = N_;
  static constexpr int NS = 4;            // states per lane
  static constexpr int G = N / NS;        // lanes per channel
  static constexpr bool GATE = GATE_;
  static constexpr bool VEC = VEC_;
  static constexpr int THREADS = 256;
};

template <typename IO, typename Cfg>
__global__ void __launch_bounds__(Cfg::THREADS) state_update_kernel(const UpdateParams p) {
  constexpr int N = Cfg::N, NS = Cfg::NS, G = Cfg::G;
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * Cfg::THREADS + threadIdx.x;
  const int64_t ch = gt / G;
  const int g = static_cast<int>(gt % G);
  const bool valid = ch < p.channels;
  const int64_t chc = valid ? ch : 0;  // clamped for address arithmetic only
  const int64_t b = chc / p.dim;
  const int d = static_cast<int>(chc % p.dim);

  float hv[NS], Av[NS], Bv[NS], Cv[NS];
  float* hp = p.h + chc * N + g * NS;
  const float* Ap = p.A + static_cast<int64_t>(d) * N + g * NS;
  const IO* Bp = static_cast<const IO*>(p.B) + b * N + g * NS;
  const IO* Cp = static_cast<const IO*>(p.C) + b * N + g * NS;
  float uv = 0.f, dv = 0.f, zv = 0.f;
  if (valid) {
    if constexpr (Cfg::VEC) {
      const float4 h4 = *reinterpret_cast<const float4*>(hp);
      const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ap));
      hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
      Av[0] = a4.x; Av[1] = a4.y; Av[2] = a4.z; Av[3] = a4.w;
      if constexpr (sizeof(IO) == 2) {
        const uint2 bw = __ldg(reinterpret_cast<const uint2*>(Bp));
        const uint2 cw = __ldg(reinterpret_cast<const uint2*>(Cp));
        Bv[0] = bf16lo(bw.x); Bv[1] = bf16hi(bw.x); Bv[2] = bf16lo(bw.y); Bv[3] = bf16hi(bw.y);
        Cv[0] = bf16lo(cw.x); Cv[1] = bf16hi(cw.x); Cv[2] = bf16lo(cw.y); Cv[3] = bf16hi(cw.y);
      } else {
        const float4 bw = __ldg(reinterpret_cast<const float4*>(Bp));
        const float4 cw = __ldg(reinterpret_cast<const float4*>(Cp));
        Bv[0] = bw.x; Bv[1] = bw.y; Bv[2] = bw.z; Bv[3] = bw.w;
        Cv[0] = cw.x; Cv[1] = cw.y; Cv[2] = cw.z; Cv[3] = cw.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        hv[i] = hp[i];
        Av[i] = __ldg(Ap + i);
        Bv[i] = Io<IO>::ldg(Bp + i);
        Cv[i] = Io<IO>::ldg(Cp + i);
      }
    }
    uv = Io<IO>::ldg(static_cast<const IO*>(p.u) + chc);
    dv = Io<IO>::ldg(static_cast<const IO*>(p.delta) + chc);
    if constexpr (Cfg::GATE) zv = Io<IO>::ldg(static_cast<const IO*>(p.z) + chc);
  } else {
#pragma unroll
    for (int i = 0; i < NS; ++i) { hv[i] = 0.f; Av[i] = -1.f; Bv[i] = 0.f; Cv[i] = 0.f; }
  }
  const float x2 = fmaf(dv, kLog2e, p.bias ? __ldg(p.bias + d) * kLog2e : 0.0f);
  const float s = p.softplus ? softplus_log2_accurate(x2) : x2;  // dt * log2(e)
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float a0 = Av[i];
    const float q = s * a0;
    const float ahw = ex2(q);
    const float em1 = exp2m1_accurate(q, ahw);
    const float abar = (fabsf(q) < 0.36f) ? 1.0f + em1 : ahw;
    const float coef = (a0 == 0.0f) ? s * kLn2 : em1 / a0;
    hv[i] = fmaf(abar, hv[i], coef * (Bv[i] * uv));
    acc = fmaf(Cv[i], hv[i], acc);
  }
#pragma unroll
  for (int o = G / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (valid) {
    if constexpr (Cfg::VEC) {
      *reinterpret_cast<float4*>(hp) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    } else {
#pragma unroll
      for (int i = 0; i < NS; ++i) hp[i] = hv[i];
    }
    if (g == 0) {
      float yv = fmaf(p.D ? __ldg(p.D + d) : 0.0f, uv, acc);
      if constexpr (Cfg::GATE) yv *= silu_accurate(zv);
      Io<IO>::store(static_cast<IO*>(p.y) + chc, yv);
    }
  }
}

}  // namespace ssm
