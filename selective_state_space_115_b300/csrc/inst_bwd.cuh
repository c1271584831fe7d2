// inst_bwd.cuh -- launches of the scan-gradient kernels, instantiated per io type
// by inst_bwd_bf16.cu and inst_bwd_f32.cu.
#pragma once

#include "ssm_host.cuh"

namespace ssm_host {

// `overlap`: launched with programmatic stream serialisation, so that it may start
// while the previous launch (the accurate CTAs) still runs
template <typename Cfg, int MODE, bool PRE>
static ssm_status bwd_launch(const ssm::BwdParams& p, cudaStream_t s, bool overlap = false) {
  auto kern = ssm::scan_bwd_kernel<Cfg, MODE, PRE>;
  // per call: the attribute belongs to the current device's context
  const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (attr != cudaSuccess) return cuda_fail(attr, "scan_bwd smem attribute");
  const int64_t grid = static_cast<int64_t>(p.nseg) * p.batch * p.tiles;
  if (grid > INT32_MAX) return SSM_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = overlap ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return cuda_fail(e, "scan_bwd launch");
  return SSM_OK;
}

// one pass (PRE: the segments' first pass) of every CTA.  bf16 ZOH: the CTAs that
// need the series coefficients (small |A| or vanishing steps, per the classify
// kernel's flags) run in the first launch, which lets the second (the fast
// coefficients, compiled apart for its lower register count) start at once; the
// second's block 0 waits for the first before it exits, so whatever follows on the
// stream sees both.
template <typename Cfg, bool PRE>
static ssm_status bwd_pass(const ssm::BwdParams& p, cudaStream_t s) {
  if constexpr (sizeof(typename Cfg::io_t) == 2 && !Cfg::EULER) {
    const ssm_status st = bwd_launch<Cfg, ssm::kBwdAccurateTiles, PRE>(p, s);
    if (st != SSM_OK) return st;
    return bwd_launch<Cfg, ssm::kBwdFastTiles, PRE>(p, s, true);
  } else {
    return bwd_launch<Cfg, ssm::kBwdAll, PRE>(p, s);
  }
}

template <typename IO, int N, bool GATE, bool EULER, bool VEC>
static ssm_status bwd_main(const ssm::BwdParams& p, cudaStream_t s) {
  using Cfg = ssm::BwdCfg<IO, N, GATE, EULER, VEC, kBwdThreads>;
  if constexpr (sizeof(IO) == 2 && !EULER) {
    const int64_t grid = static_cast<int64_t>(p.nseg) * p.batch * p.tiles;
    ssm::scan_bwd_classify_kernel<N><<<static_cast<unsigned>(grid), 128, 0, s>>>(
        p, VEC, const_cast<unsigned char*>(p.cta_fast));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd classify launch");
  }
  if (p.nseg > 1) {
    const ssm_status st = bwd_pass<Cfg, true>(p, s);
    if (st != SSM_OK) return st;
  }
  return bwd_pass<Cfg, false>(p, s);
}

template <typename IO, int N>
static ssm_status bwd_main_n(const ssm::BwdParams& p, bool gate, bool euler, bool vec,
                             cudaStream_t s) {
  if (gate) {
    if (euler) return vec ? bwd_main<IO, N, true, true, true>(p, s) : bwd_main<IO, N, true, true, false>(p, s);
    return vec ? bwd_main<IO, N, true, false, true>(p, s) : bwd_main<IO, N, true, false, false>(p, s);
  }
  if (euler) return vec ? bwd_main<IO, N, false, true, true>(p, s) : bwd_main<IO, N, false, true, false>(p, s);
  return vec ? bwd_main<IO, N, false, false, true>(p, s) : bwd_main<IO, N, false, false, false>(p, s);
}

template <typename IO>
ssm_status launch_scan_bwd(const ssm::BwdParams& p, int dstate, bool gate, bool euler, bool vec,
                           void* dB, void* dC, float* dA, float* dD, float* dbias,
                           cudaStream_t s) {
  ssm_status st = SSM_OK;
  if (p.batch * p.dim > 0) {
    switch (dstate) {
      case 4: st = bwd_main_n<IO, 4>(p, gate, euler, vec, s); break;
      case 8: st = bwd_main_n<IO, 8>(p, gate, euler, vec, s); break;
      case 16: st = bwd_main_n<IO, 16>(p, gate, euler, vec, s); break;
      default: return SSM_ERR_UNSUPPORTED;
    }
    if (st != SSM_OK) return st;
  }
  const int64_t nbc = p.batch * 2 * dstate * static_cast<int64_t>(p.seqlen);
  if (nbc > 0) {
    ssm::scan_bwd_reduce_bc_kernel<IO><<<static_cast<unsigned>((nbc + 255) / 256), 256, 0, s>>>(
        p.part_bc, p.tiles, p.batch, dstate, p.seqlen, static_cast<IO*>(dB), static_cast<IO*>(dC));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd reduce launch");
  }
  const int64_t npar = static_cast<int64_t>(p.dim) * dstate + p.dim;
  if (npar > 0) {
    // the partials are [nseg][batch][dim]: sum over nseg * batch row blocks
    ssm::scan_bwd_reduce_param_kernel<><<<static_cast<unsigned>((npar + 255) / 256), 256, 0, s>>>(
        p.part_a, p.part_dd, p.batch * p.nseg, p.dim, dstate, dA, dD, dbias);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd reduce launch");
  }
  return SSM_OK;
}

}  // namespace ssm_host
