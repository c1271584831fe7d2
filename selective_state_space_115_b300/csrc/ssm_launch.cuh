// ssm_launch.cuh -- kernel launchers of libssm (TMA descriptors, grids, shared
// memory) and the per-type dispatchers.  Included only by the inst_*.cu
// translation units, each of which instantiates a share of the dispatchers, so
// the kernels compile in parallel.
#pragma once

#include "ssm_host.cuh"
#include "scan_chunk.cuh"

namespace ssm_host {

// The channel-kernel instantiation a pass runs: y only (the plain forward), y and the
// state checkpoints (the training forward), or the checkpoints alone (the gradient's
// own forward: a call without y, and without the gate, whose z it would not read).
template <typename IO, typename Cfg, int MODE>
static auto chan_kernel(const ScanCall& c, const ScanParams& p) {
  if constexpr (!Cfg::GATE) {
    if (!c.y) return ssm::scan_channel_kernel<IO, Cfg, MODE, true, false>;
  }
  return p.ckpt ? ssm::scan_channel_kernel<IO, Cfg, MODE, true, true>
                : ssm::scan_channel_kernel<IO, Cfg, MODE, false, true>;
}

template <typename IO, int N, bool GATE, int LPC, bool EULER>
ssm_status launch_channel(const ScanCall& c, void* workspace, cudaStream_t stream,
                          const SegPlan& seg = SegPlan()) {
  using Shape = ChanShape<LPC>;
  using Cfg = ChanCfg<IO, N, GATE, LPC, Shape::S, Shape::RB, EULER>;
  ChanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const bool bf = c.bf16;
  const uint64_t L = c.seqlen, Dm = c.dim, Bt = c.batch, Nn = N;
  if (!make_map(&maps.u, c.u, bf, L, Dm, Bt, Cfg::LC, Cfg::DT) ||
      !make_map(&maps.delta, c.delta, bf, L, Dm, Bt, Cfg::LC, Cfg::DT) ||
      !make_map(&maps.B, c.B, bf, L, Nn, Bt, Cfg::LC, N) ||
      !make_map(&maps.C, c.C, bf, L, Nn, Bt, Cfg::LC, N) ||
      (GATE && !make_map(&maps.z, c.z, bf, L, Dm, Bt, Cfg::LC, Cfg::DT))) {
    g_last_cuda_error = "cuTensorMapEncodeTiled failed";
    return SSM_ERR_CUDA;
  }
  ScanParams p = make_params(c, workspace);
  if (!c.y && (GATE || !p.ckpt)) return SSM_ERR_INVALID_ARG;  // a pass writes y or checkpoints
  p.dtiles = static_cast<int>((c.dim + Cfg::DT - 1) / Cfg::DT);
  const int64_t tiles = c.batch * p.dtiles;
  if (tiles * (seg.nseg > 1 ? seg.nseg : 1) > INT32_MAX) return SSM_ERR_INVALID_ARG;
  if constexpr (LPC == 1) {
    if (seg.nseg > 1) {
      // pass 1 (segments 0 .. nseg-2: each segment's end state from h = 0 and its
      // step-size sum), then pass 2 (every segment, entering state rebuilt from them)
      p.nseg = seg.nseg;
      p.seg_len = seg.seg_len;
      const size_t chans = static_cast<size_t>(c.batch) * static_cast<size_t>(c.dim);
      uint8_t* base = static_cast<uint8_t*>(workspace);
      p.seg_state = reinterpret_cast<float*>(base + kStatusBytes);
      p.seg_sum = reinterpret_cast<float*>(
          base + kStatusBytes + round_up(static_cast<size_t>(seg.nseg) * chans * N * 4, 256));
      auto k1 = ssm::scan_channel_kernel<IO, Cfg, ssm::kModeStates>;
      auto k2 = chan_kernel<IO, Cfg, ssm::kModeCarry>(c, p);
      cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg::SMEM_ALLOC);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(scan_channel)");
      k1<<<static_cast<unsigned>(tiles * (seg.nseg - 1)), Cfg::THREADS, Cfg::SMEM_ALLOC, stream>>>(
          maps, p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "scan_channel (segment states) launch");
      k2<<<static_cast<unsigned>(tiles * seg.nseg), Cfg::THREADS, Cfg::SMEM_ALLOC, stream>>>(maps,
                                                                                               p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "scan_channel (segments) launch");
      return SSM_OK;
    }
  }
  auto kern = chan_kernel<IO, Cfg, ssm::kModeFull>(c, p);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(scan_channel)");
  kern<<<static_cast<unsigned>(tiles), Cfg::THREADS, Cfg::SMEM_ALLOC, stream>>>(maps, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_channel launch");
  return SSM_OK;
}

template <typename IO, bool GATE, bool EULER>
ssm_status launch_mixed(const ScanCall& c, void* workspace, cudaStream_t stream,
                        const MixPlan& m) {
  using CfgA = ChanCfg<IO, 16, GATE, 1, ChanShape<1>::S, ChanShape<1>::RB, EULER>;
  using CfgB = ChanCfg<IO, 16, GATE, 4, ChanShape<4>::S, ChanShape<4>::RB, EULER>;
  static_assert(CfgA::LC == CfgB::LC, "one chunk width for both roles");
  ChanMaps ma, mb;
  std::memset(&ma, 0, sizeof(ma));
  std::memset(&mb, 0, sizeof(mb));
  const bool bf = c.bf16;
  const uint64_t L = c.seqlen, Dm = c.dim, Bt = c.batch, Nn = 16;
  bool ok = true;
  for (int r = 0; r < 2 && ok; ++r) {
    ChanMaps& mp = r ? mb : ma;
    const uint32_t rows = r ? CfgB::DT : CfgA::DT;
    ok = make_map(&mp.u, c.u, bf, L, Dm, Bt, CfgA::LC, rows) &&
         make_map(&mp.delta, c.delta, bf, L, Dm, Bt, CfgA::LC, rows) &&
         make_map(&mp.B, c.B, bf, L, Nn, Bt, CfgA::LC, 16) &&
         make_map(&mp.C, c.C, bf, L, Nn, Bt, CfgA::LC, 16) &&
         (!GATE || make_map(&mp.z, c.z, bf, L, Dm, Bt, CfgA::LC, rows));
  }
  if (!ok) {
    g_last_cuda_error = "cuTensorMapEncodeTiled failed";
    return SSM_ERR_CUDA;
  }
  ScanParams p = make_params(c, workspace);
  ssm::MixSched sched;
  sched.k = m.k;
  sched.n_tiles = m.n_tiles;
  sched.n_quarters = m.n_quarters;
  sched.dtiles128 = m.dtiles128;
  sched.counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  sched.max_sm_slots = static_cast<unsigned>(kMixCounterBytes / sizeof(unsigned) - 2);
  cudaError_t e = cudaMemsetAsync(sched.counters, 0, kMixCounterBytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scheduler counters)");
  constexpr int smem = CfgA::SMEM_ALLOC > CfgB::SMEM_ALLOC ? CfgA::SMEM_ALLOC : CfgB::SMEM_ALLOC;
  if (!c.y && (GATE || !p.ckpt)) return SSM_ERR_INVALID_ARG;  // a pass writes y or checkpoints
  auto kern = p.ckpt ? ssm::scan_channel_mixed_kernel<IO, CfgA, CfgB, true, true>
                     : ssm::scan_channel_mixed_kernel<IO, CfgA, CfgB, false, true>;
  if constexpr (!GATE) {
    if (!c.y) kern = ssm::scan_channel_mixed_kernel<IO, CfgA, CfgB, true, false>;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(scan_channel_mixed)");
  const unsigned grid = static_cast<unsigned>(m.n_tiles + m.n_quarters);
  kern<<<grid, CfgA::THREADS, smem, stream>>>(ma, mb, p, sched);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_channel_mixed launch");
  return SSM_OK;
}

template <typename IO, int N, bool GATE, bool VEC, bool EULER>
ssm_status launch_chunk(const ScanCall& c, void* workspace, cudaStream_t stream) {
  using Cfg = ChunkCfg<IO, N, GATE, VEC, EULER>;
  ScanParams p = make_params(c, workspace);
  // one CTA per (batch row, group of WARPS channels)
  const int64_t grid64 = c.batch * ((c.dim + Cfg::WARPS - 1) / Cfg::WARPS);
  if (grid64 > INT32_MAX) return SSM_ERR_INVALID_ARG;
  auto kern =
      p.ckpt ? ssm::scan_chunk_kernel<IO, Cfg, true> : ssm::scan_chunk_kernel<IO, Cfg, false>;
  // per call: the attribute belongs to the current device's context
  const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (attr != cudaSuccess) return cuda_fail(attr, "scan_chunk smem attribute");
  kern<<<static_cast<unsigned>(grid64), Cfg::THREADS, Cfg::SMEM, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_chunk launch");
  return SSM_OK;
}

template <typename IO, int N, int LPC, bool EULER>
ssm_status launch_channel_lpc(const ScanCall& c, void* ws, cudaStream_t s) {
  if constexpr (N / LPC >= 4) {
    return c.z ? launch_channel<IO, N, true, LPC, EULER>(c, ws, s)
               : launch_channel<IO, N, false, LPC, EULER>(c, ws, s);
  } else {
    return SSM_ERR_UNSUPPORTED;
  }
}

template <typename IO, int N, bool EULER>
ssm_status dispatch_scan_n(const ScanCall& c, ssm_algo algo, void* ws, cudaStream_t s,
                           const SegPlan& seg, const MixPlan& mix) {
  const bool gate = c.z != nullptr;
  if constexpr (N == 16) {
    if (algo == SSM_ALGO_CHANNEL_MIXED)
      return gate ? launch_mixed<IO, true, EULER>(c, ws, s, mix)
                  : launch_mixed<IO, false, EULER>(c, ws, s, mix);
  }
  if (algo == SSM_ALGO_SEGMENTED) {
    return gate ? launch_channel<IO, N, true, 1, EULER>(c, ws, s, seg)
                : launch_channel<IO, N, false, 1, EULER>(c, ws, s, seg);
  }
  if (algo == SSM_ALGO_CHANNEL) {
    switch (choose_lpc(c.batch, c.dim, N)) {
      case 4: return launch_channel_lpc<IO, N, 4, EULER>(c, ws, s);
      case 2: return launch_channel_lpc<IO, N, 2, EULER>(c, ws, s);
      default: return launch_channel_lpc<IO, N, 1, EULER>(c, ws, s);
    }
  }
  if (algo == SSM_ALGO_CHANNEL_L1) return launch_channel_lpc<IO, N, 1, EULER>(c, ws, s);
  if (algo == SSM_ALGO_CHANNEL_L2) return launch_channel_lpc<IO, N, 2, EULER>(c, ws, s);
  if (algo == SSM_ALGO_CHANNEL_L4) return launch_channel_lpc<IO, N, 4, EULER>(c, ws, s);
  if (vec_eligible(c))
    return gate ? launch_chunk<IO, N, true, true, EULER>(c, ws, s)
                : launch_chunk<IO, N, false, true, EULER>(c, ws, s);
  return gate ? launch_chunk<IO, N, true, false, EULER>(c, ws, s)
              : launch_chunk<IO, N, false, false, EULER>(c, ws, s);
}

template <typename IO, int N, bool GATE, bool VEC, bool EULER>
ssm_status launch_update(const UpdateParams& p0, cudaStream_t stream) {
  using Cfg = UpdCfg<IO, N, GATE, VEC, EULER>;
  // one lane per channel: x over blocks of a batch row, y over up to 65535 batch rows
  // per launch
  constexpr int64_t kRowsPerLaunch = 65535;
  UpdateParams p = p0;
  for (int64_t b0 = 0; b0 < p0.batch; b0 += kRowsPerLaunch) {
    p.b0 = b0;
    const int64_t rows = (p0.batch - b0 < kRowsPerLaunch) ? p0.batch - b0 : kRowsPerLaunch;
    const dim3 grid(static_cast<unsigned>((p.dim + Cfg::THREADS - 1) / Cfg::THREADS),
                    static_cast<unsigned>(rows));
    // programmatic stream serialisation: consecutive decode steps overlap the next
    // step's launch with this one's last wave (the kernel waits for its
    // predecessor before reading anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, ssm::state_update_kernel<IO, Cfg>, p);
    if (e != cudaSuccess) return cuda_fail(e, "state_update launch");
  }
  return SSM_OK;
}

template <typename IO, int N, bool EULER>
ssm_status dispatch_update_n(const UpdateParams& p, bool vec, cudaStream_t s) {
  const bool gate = p.z != nullptr;
  if (vec)
    return gate ? launch_update<IO, N, true, true, EULER>(p, s)
                : launch_update<IO, N, false, true, EULER>(p, s);
  return gate ? launch_update<IO, N, true, false, EULER>(p, s)
              : launch_update<IO, N, false, false, EULER>(p, s);
}

}  // namespace ssm_host
