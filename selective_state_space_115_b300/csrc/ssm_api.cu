// ssm_api.cu -- C ABI of libssm (declared in include/ssm.h).
//
// Host side: argument validation (nothing is enqueued when it fails), choice of
// kernel family, TMA descriptor encoding, launches on the caller's stream.
// The library allocates no device memory and keeps no per-call state.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "ssm.h"
#include "scan_channel.cuh"
#include "scan_chunk.cuh"
#include "state_update.cuh"

namespace {

using ssm::ChanCfg;
using ssm::ChanMaps;
using ssm::ChunkCfg;
using ssm::ScanParams;
using ssm::UpdateParams;
using ssm::UpdCfg;

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr size_t kWorkspaceBytes = 256;
// channel kernel only when there are enough (batch, dim) channels to fill the GPU
// with lanes-over-channels warps; below this the chunk kernel's lanes-over-positions
// layout keeps every SM busy.
constexpr int64_t kChannelKernelMinChannels = 8192;

thread_local std::string g_last_cuda_error;

ssm_status cuda_fail(cudaError_t e, const char* what) {
  g_last_cuda_error = std::string(what) + ": " + cudaGetErrorString(e);
  return SSM_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// TMA descriptor encoding through the driver entry point
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 3-D map over a [d2][d1][d0] tensor (d0 fastest), box {box0, box1, 1}, zero fill
// outside the tensor.  The box row (box0 elements) must be exactly one swizzle
// span (32, 64 or 128 bytes): the kernels index their tiles with that span's
// XOR pattern and size them for rows of exactly that width.
bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t box0, uint32_t box1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint64_t esz = bf16 ? 2 : 4;
  CUtensorMapSwizzle swz;
  switch (box0 * esz) {
    case 32: swz = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: swz = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: swz = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
  }
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esz, d0 * d1 * esz};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
struct ScanCall {
  int64_t batch, dim, dstate, seqlen;
  bool bf16;
  const void *u, *delta, *B, *C, *z;
  const float *bias, *A, *D, *h0;
  float* h_last;
  void* y;
  int softplus;
};

ssm_status validate_common(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io) {
  if (batch < 1 || dim < 1 || dstate < 1) return SSM_ERR_INVALID_ARG;
  if (io != SSM_DTYPE_F32 && io != SSM_DTYPE_BF16) return SSM_ERR_UNSUPPORTED;
  if (dstate != 4 && dstate != 8 && dstate != 16) return SSM_ERR_UNSUPPORTED;
  if (dim > INT32_MAX || batch > INT32_MAX) return SSM_ERR_INVALID_ARG;
  return SSM_OK;
}

ssm_status validate_scan(const ScanCall& c, const void* workspace, size_t workspace_bytes) {
  ssm_status st = validate_common(c.batch, c.dim, c.dstate, c.bf16 ? SSM_DTYPE_BF16 : SSM_DTYPE_F32);
  if (st != SSM_OK) return st;
  if (c.seqlen < 1 || c.seqlen > INT32_MAX - 4096) return SSM_ERR_INVALID_ARG;
  // element counts must fit comfortably in 63 bits
  if (c.batch > (int64_t(1) << 62) / c.dim / c.seqlen) return SSM_ERR_INVALID_ARG;
  if (!c.u || !c.delta || !c.A || !c.B || !c.C || !c.y || !workspace) return SSM_ERR_INVALID_ARG;
  const size_t esz = c.bf16 ? 2 : 4;
  const void* io_ptrs[6] = {c.u, c.delta, c.B, c.C, c.y, c.z};
  for (const void* q : io_ptrs)
    if (q && !aligned(q, esz)) return SSM_ERR_INVALID_ARG;
  const float* f_ptrs[5] = {c.A, c.D, c.bias, c.h0, c.h_last};
  for (const float* q : f_ptrs)
    if (q && !aligned(q, 4)) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 16) || workspace_bytes < kWorkspaceBytes) return SSM_ERR_INVALID_ARG;
  // the chunk kernel's grid has one CTA per 4 channels
  if ((c.batch * c.dim + 3) / 4 > INT32_MAX) return SSM_ERR_INVALID_ARG;
  return SSM_OK;
}

bool tma_eligible(const ScanCall& c) {
  const int64_t esz = c.bf16 ? 2 : 4;
  if ((c.seqlen * esz) % 16 != 0) return false;
  const void* ptrs[6] = {c.u, c.delta, c.B, c.C, c.y, c.z};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return false;
  return encode_fn() != nullptr;
}

bool vec_eligible(const ScanCall& c) {
  const int64_t esz = c.bf16 ? 2 : 4;
  if ((c.seqlen * esz) % 16 != 0) return false;
  const void* ptrs[6] = {c.u, c.delta, c.B, c.C, c.y, c.z};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return false;
  return true;
}

// SM count of the current device (cached per device ordinal).
int sm_count() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

ScanParams make_params(const ScanCall& c, void* workspace) {
  ScanParams p;
  p.batch = static_cast<int>(c.batch);
  p.dim = static_cast<int>(c.dim);
  p.seqlen = static_cast<int>(c.seqlen);
  p.dtiles = 1;
  p.softplus = c.softplus;
  p.A = c.A;
  p.D = c.D;
  p.bias = c.bias;
  p.h0 = c.h0;
  p.h_last = c.h_last;
  p.status = static_cast<ssm::DeviceStatus*>(workspace);
  p.u = c.u;
  p.delta = c.delta;
  p.z = c.z;
  p.B = c.B;
  p.C = c.C;
  p.y = c.y;
  p.nseg = 1;
  p.seg_len = static_cast<int>(c.seqlen);
  p.seg_state = nullptr;
  p.seg_sum = nullptr;
  return p;
}

// ---------------------------------------------------------------------------
// segmented (two-pass) plan for long sequences over few channels
// ---------------------------------------------------------------------------
// Workspace layout: [0, 256) device status words; then the segments' end states
// [nseg][batch * dim][N] fp32; then their step-size sums [nseg][batch * dim] fp32.
constexpr size_t kStatusBytes = 256;
constexpr int64_t kSegMinLen = 256;        // positions: shorter segments cost more than they gain
constexpr int64_t kSegMinSeqlen = 8192;    // AUTO splits sequences at least this long
constexpr int kSegCtasPerSm = 3;            // one-lane-per-channel CTAs an SM holds at once

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SegPlan {
  int nseg = 1;     // 1: not segmented
  int seg_len = 0;
};

// Segments for the one-lane-per-channel channel kernel: enough that the CTAs fill
// every SM (kSegCtasPerSm per SM), each at least kSegMinLen positions long, a
// multiple of the chunk (lc positions).  `force` asks for at least two segments.
SegPlan seg_plan(int64_t batch, int64_t dim, int64_t seqlen, int lc, bool force) {
  SegPlan pl;
  const int64_t ctas = batch * ((dim + 127) / 128);
  int64_t nseg = static_cast<int64_t>(sm_count()) * kSegCtasPerSm / ctas;
  if (nseg > seqlen / kSegMinLen) nseg = seqlen / kSegMinLen;
  if (force && nseg < 2) nseg = 2;
  if (nseg > (seqlen + lc - 1) / lc) nseg = (seqlen + lc - 1) / lc;
  if (nseg < 2) return pl;
  int64_t len = (seqlen + nseg - 1) / nseg;
  len = (len + lc - 1) / lc * lc;
  pl.nseg = static_cast<int>((seqlen + len - 1) / len);
  pl.seg_len = static_cast<int>(len);
  if (pl.nseg < 2) pl.nseg = 1;
  return pl;
}

size_t seg_workspace_bytes(int64_t batch, int64_t dim, int64_t dstate, const SegPlan& pl) {
  if (pl.nseg < 2) return kStatusBytes;
  const size_t chans = static_cast<size_t>(batch) * static_cast<size_t>(dim);
  return kStatusBytes + round_up(static_cast<size_t>(pl.nseg) * chans * dstate * 4, 256) +
         round_up(static_cast<size_t>(pl.nseg) * chans * 4, 256);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Channel-kernel shapes: 32-byte chunk rows (16 bf16 / 8 fp32 positions) and a
// 4-stage ring.  Per 4-warp CTA (bf16, dstate 16, gate): ~66 KB of shared memory
// and ~107 registers a thread at 1 lane per channel (3 CTAs per SM), ~37 KB and
// ~80 at 2 (6 per SM), ~22 KB and ~56 at 4 (9 per SM).
template <int LPC>
struct ChanShape {
  static constexpr int S = 4, RB = 32;
};

template <typename IO, int N, bool GATE, int LPC>
ssm_status launch_channel(const ScanCall& c, void* workspace, cudaStream_t stream,
                          const SegPlan& seg = SegPlan()) {
  using Shape = ChanShape<LPC>;
  using Cfg = ChanCfg<IO, N, GATE, LPC, Shape::S, Shape::RB>;
  ChanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const bool bf = c.bf16;
  const uint64_t L = c.seqlen, Dm = c.dim, Bt = c.batch, Nn = N;
  if (!make_map(&maps.u, c.u, bf, L, Dm, Bt, Cfg::LC, Cfg::DT) ||
      !make_map(&maps.delta, c.delta, bf, L, Dm, Bt, Cfg::LC, Cfg::DT) ||
      !make_map(&maps.y, c.y, bf, L, Dm, Bt, Cfg::LC, Cfg::DT) ||
      !make_map(&maps.B, c.B, bf, L, Nn, Bt, Cfg::LC, N) ||
      !make_map(&maps.C, c.C, bf, L, Nn, Bt, Cfg::LC, N) ||
      (GATE && !make_map(&maps.z, c.z, bf, L, Dm, Bt, Cfg::LC, Cfg::DT))) {
    g_last_cuda_error = "cuTensorMapEncodeTiled failed";
    return SSM_ERR_CUDA;
  }
  ScanParams p = make_params(c, workspace);
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
      auto k2 = ssm::scan_channel_kernel<IO, Cfg, ssm::kModeCarry>;
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
  auto kern = ssm::scan_channel_kernel<IO, Cfg, ssm::kModeFull>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(scan_channel)");
  kern<<<static_cast<unsigned>(tiles), Cfg::THREADS, Cfg::SMEM_ALLOC, stream>>>(maps, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_channel launch");
  return SSM_OK;
}

// Lanes per channel for the channel kernel.  Every SM sub-partition runs one warp
// of each resident CTA, so the busiest sub-partition processes kmax = ceil(CTAs /
// SMs) warps.  Its time is the larger of kmax x the issue cost of one warp (which
// falls with the states a lane holds, NS = dstate / LPC, but less than in
// proportion because the per-position work and the lane exchange do not shrink)
// and the latency of a single warp when there are too few warps to overlap.  The
// relative costs below were measured on B300 with the 2.8B-like layer (bf16,
// dstate 16, L 2048): one warp of NS = 16 / 8 / 4 states costs 1 / 0.58 / 0.37
// when sub-partitions are full, and a lone warp takes 1.78 / 1.6 / 1.2.
int choose_lpc(int64_t batch, int64_t dim, int64_t dstate, double* cost_out = nullptr) {
  const int64_t sms = sm_count();
  int best = 1;
  double best_cost = 0.0;
  for (int lpc = 1; lpc <= 4; lpc *= 2) {
    const int64_t ns = dstate / lpc;
    if (ns < 4) break;
    const double w = (ns >= 16) ? 1.0 : (ns >= 8) ? 0.58 : 0.37;
    const double lone = (ns >= 16) ? 1.78 : (ns >= 8) ? 1.6 : 1.2;
    const int64_t dt = 128 / lpc;
    const int64_t ctas = batch * ((dim + dt - 1) / dt);
    const double kmax = double((ctas + sms - 1) / sms);
    const double cost = (kmax * w > lone) ? kmax * w : lone;
    if (lpc == 1 || cost < best_cost) {
      best = lpc;
      best_cost = cost;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best;
}

// Mixed split (dstate 16): k = floor(T / SMs) one-lane CTAs per SM for T 128-channel
// tiles, the remaining tiles as 32-channel four-lane CTAs.  In the units of the model
// above its busiest sub-partition costs k x 1 + ceil(quarters / SMs) x 0.37.
// Scheduler counters live in the workspace after the status words.
constexpr size_t kMixCounterBytes = 1280;  // [2 + SMs] unsigned, up to 318 SMs
constexpr int kMixMaxSms = 318;

struct MixPlan {
  bool use = false;
  int k = 0, n_tiles = 0, n_quarters = 0, dtiles128 = 0;
};

MixPlan mix_plan(int64_t batch, int64_t dim) {
  MixPlan m;
  const int64_t sms = sm_count();
  const int64_t dt = (dim + 127) / 128;
  const int64_t tiles = batch * dt;
  if (sms > kMixMaxSms || tiles * 4 > INT32_MAX) return m;
  m.k = static_cast<int>(tiles / sms);
  if (m.k > 2) m.k = 2;  // three 66 KB CTAs fill an SM's shared memory
  m.n_tiles = static_cast<int>(m.k * sms);
  m.n_quarters = static_cast<int>((tiles - m.n_tiles) * 4);
  m.dtiles128 = static_cast<int>(dt);
  m.use = true;
  return m;
}

double mix_cost(const MixPlan& m) {
  const int64_t sms = sm_count();
  return m.k * 1.0 + double((m.n_quarters + sms - 1) / sms) * 0.37;
}

template <typename IO, bool GATE>
ssm_status launch_mixed(const ScanCall& c, void* workspace, cudaStream_t stream,
                        const MixPlan& m) {
  using CfgA = ChanCfg<IO, 16, GATE, 1, ChanShape<1>::S, ChanShape<1>::RB>;
  using CfgB = ChanCfg<IO, 16, GATE, 4, ChanShape<4>::S, ChanShape<4>::RB>;
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
         make_map(&mp.y, c.y, bf, L, Dm, Bt, CfgA::LC, rows) &&
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
  auto kern = ssm::scan_channel_mixed_kernel<IO, CfgA, CfgB>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(scan_channel_mixed)");
  const unsigned grid = static_cast<unsigned>(m.n_tiles + m.n_quarters);
  kern<<<grid, CfgA::THREADS, smem, stream>>>(ma, mb, p, sched);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_channel_mixed launch");
  return SSM_OK;
}

template <typename IO, int N, bool GATE, bool VEC>
ssm_status launch_chunk(const ScanCall& c, void* workspace, cudaStream_t stream) {
  using Cfg = ChunkCfg<IO, N, GATE, VEC>;
  ScanParams p = make_params(c, workspace);
  const int64_t channels = c.batch * c.dim;
  const unsigned grid = static_cast<unsigned>((channels + Cfg::WARPS - 1) / Cfg::WARPS);
  ssm::scan_chunk_kernel<IO, Cfg><<<grid, Cfg::THREADS, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan_chunk launch");
  return SSM_OK;
}

template <typename IO, int N, int LPC>
ssm_status launch_channel_lpc(const ScanCall& c, void* ws, cudaStream_t s) {
  if constexpr (N / LPC >= 4) {
    return c.z ? launch_channel<IO, N, true, LPC>(c, ws, s)
               : launch_channel<IO, N, false, LPC>(c, ws, s);
  } else {
    return SSM_ERR_UNSUPPORTED;
  }
}

template <typename IO, int N>
ssm_status dispatch_scan_n(const ScanCall& c, ssm_algo algo, void* ws, cudaStream_t s,
                           const SegPlan& seg, const MixPlan& mix) {
  const bool gate = c.z != nullptr;
  if constexpr (N == 16) {
    if (algo == SSM_ALGO_CHANNEL_MIXED)
      return gate ? launch_mixed<IO, true>(c, ws, s, mix) : launch_mixed<IO, false>(c, ws, s, mix);
  }
  if (algo == SSM_ALGO_SEGMENTED) {
    return gate ? launch_channel<IO, N, true, 1>(c, ws, s, seg)
                : launch_channel<IO, N, false, 1>(c, ws, s, seg);
  }
  if (algo == SSM_ALGO_CHANNEL) {
    switch (choose_lpc(c.batch, c.dim, N)) {
      case 4: return launch_channel_lpc<IO, N, 4>(c, ws, s);
      case 2: return launch_channel_lpc<IO, N, 2>(c, ws, s);
      default: return launch_channel_lpc<IO, N, 1>(c, ws, s);
    }
  }
  if (algo == SSM_ALGO_CHANNEL_L1) return launch_channel_lpc<IO, N, 1>(c, ws, s);
  if (algo == SSM_ALGO_CHANNEL_L2) return launch_channel_lpc<IO, N, 2>(c, ws, s);
  if (algo == SSM_ALGO_CHANNEL_L4) return launch_channel_lpc<IO, N, 4>(c, ws, s);
  if (vec_eligible(c))
    return gate ? launch_chunk<IO, N, true, true>(c, ws, s) : launch_chunk<IO, N, false, true>(c, ws, s);
  return gate ? launch_chunk<IO, N, true, false>(c, ws, s) : launch_chunk<IO, N, false, false>(c, ws, s);
}

template <typename IO>
ssm_status dispatch_scan(const ScanCall& c, ssm_algo algo, void* ws, cudaStream_t s,
                         const SegPlan& seg, const MixPlan& mix) {
  switch (c.dstate) {
    case 4: return dispatch_scan_n<IO, 4>(c, algo, ws, s, seg, mix);
    case 8: return dispatch_scan_n<IO, 8>(c, algo, ws, s, seg, mix);
    case 16: return dispatch_scan_n<IO, 16>(c, algo, ws, s, seg, mix);
    default: return SSM_ERR_UNSUPPORTED;
  }
}

template <typename IO, int N, bool GATE, bool VEC>
ssm_status launch_update(const UpdateParams& p0, cudaStream_t stream) {
  using Cfg = UpdCfg<IO, N, GATE, VEC>;
  // one lane per channel: x over blocks of a batch row, y over up to 65535 batch rows
  // per launch
  constexpr int64_t kRowsPerLaunch = 65535;
  UpdateParams p = p0;
  for (int64_t b0 = 0; b0 < p0.batch; b0 += kRowsPerLaunch) {
    p.b0 = b0;
    const int64_t rows = (p0.batch - b0 < kRowsPerLaunch) ? p0.batch - b0 : kRowsPerLaunch;
    const dim3 grid(static_cast<unsigned>((p.dim + Cfg::THREADS - 1) / Cfg::THREADS),
                    static_cast<unsigned>(rows));
    ssm::state_update_kernel<IO, Cfg><<<grid, Cfg::THREADS, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "state_update launch");
  }
  return SSM_OK;
}

template <typename IO, int N>
ssm_status dispatch_update_n(const UpdateParams& p, bool vec, cudaStream_t s) {
  const bool gate = p.z != nullptr;
  if (vec)
    return gate ? launch_update<IO, N, true, true>(p, s) : launch_update<IO, N, false, true>(p, s);
  return gate ? launch_update<IO, N, true, false>(p, s) : launch_update<IO, N, false, false>(p, s);
}

template <typename IO>
ssm_status dispatch_update(const UpdateParams& p, int64_t dstate, bool vec, cudaStream_t s) {
  switch (dstate) {
    case 4: return dispatch_update_n<IO, 4>(p, vec, s);
    case 8: return dispatch_update_n<IO, 8>(p, vec, s);
    case 16: return dispatch_update_n<IO, 16>(p, vec, s);
    default: return SSM_ERR_UNSUPPORTED;
  }
}

// ---------------------------------------------------------------------------
// statically reserved scratch for ssm_scan_fwd_noalloc
// ---------------------------------------------------------------------------
// Device scratch of fixed size that every GPU loading this library holds until
// the process exits.  Host code must not pass the symbol itself to a kernel (on
// the host it only names a stand-in object); the device address is looked up
// once per device with cudaGetSymbolAddress.
constexpr size_t kNoAllocScratchBytes = 4096;
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the static scratch on the current device (set-up on first use).
ssm_status noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    g_last_cuda_error = "ssm_scan_fwd_noalloc: device ordinal beyond the supported range";
    return SSM_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SSM_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

size_t ssm_scan_fwd_algo_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                        int64_t seqlen, ssm_algo algo) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1) return kWorkspaceBytes;
  if (batch > (int64_t(1) << 62) / dim / seqlen) return kWorkspaceBytes;
  // the segmented plan for fp32 (8-position chunks); bf16's 16-position chunks never
  // need more segments
  // the mixed split keeps scheduler counters after the status words
  const bool many = batch * dim >= kChannelKernelMinChannels;
  if (algo == SSM_ALGO_CHANNEL_MIXED ||
      (dstate == 16 && (algo == SSM_ALGO_CHANNEL || (algo == SSM_ALGO_AUTO && many))))
    return kStatusBytes + kMixCounterBytes;
  SegPlan pl;
  if (algo == SSM_ALGO_SEGMENTED)
    pl = seg_plan(batch, dim, seqlen, 8, true);
  else if (algo == SSM_ALGO_AUTO && !many && seqlen >= kSegMinSeqlen)
    pl = seg_plan(batch, dim, seqlen, 8, false);
  return seg_workspace_bytes(batch, dim, dstate, pl);
}

size_t ssm_scan_fwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
  return ssm_scan_fwd_algo_workspace_size(batch, dim, dstate, seqlen, SSM_ALGO_AUTO);
}

ssm_status ssm_scan_fwd_algo(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             ssm_dtype io, const void* u, const void* delta,
                             const float* delta_bias, int delta_softplus, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* h0, float* h_last, void* y, void* workspace,
                             size_t workspace_bytes, ssm_algo algo, ssm_stream_t stream) {
  if (algo != SSM_ALGO_AUTO && algo != SSM_ALGO_CHANNEL && algo != SSM_ALGO_CHUNK &&
      algo != SSM_ALGO_CHANNEL_L1 && algo != SSM_ALGO_CHANNEL_L2 && algo != SSM_ALGO_CHANNEL_L4 &&
      algo != SSM_ALGO_SEGMENTED && algo != SSM_ALGO_CHANNEL_MIXED)
    return SSM_ERR_UNSUPPORTED;
  if ((algo == SSM_ALGO_CHANNEL_L2 && dstate < 8) || (algo == SSM_ALGO_CHANNEL_L4 && dstate < 16))
    return SSM_ERR_UNSUPPORTED;
  ScanCall c;
  c.batch = batch;
  c.dim = dim;
  c.dstate = dstate;
  c.seqlen = seqlen;
  c.bf16 = (io == SSM_DTYPE_BF16);
  c.u = u;
  c.delta = delta;
  c.B = B;
  c.C = C;
  c.z = z;
  c.bias = delta_bias;
  c.A = A;
  c.D = D;
  c.h0 = h0;
  c.h_last = h_last;
  c.y = y;
  c.softplus = delta_softplus ? 1 : 0;
  if (io != SSM_DTYPE_F32 && io != SSM_DTYPE_BF16) return SSM_ERR_UNSUPPORTED;
  ssm_status st = validate_scan(c, workspace, workspace_bytes);
  if (st != SSM_OK) return st;

  const int lc = c.bf16 ? 16 : 8;  // channel kernel chunk (32-byte rows)
  SegPlan seg;
  if (algo == SSM_ALGO_SEGMENTED) {
    seg = seg_plan(c.batch, c.dim, c.seqlen, lc, true);
    if (seg.nseg < 2) {
      algo = SSM_ALGO_CHANNEL_L1;  // too short to split
    } else if (workspace_bytes < seg_workspace_bytes(c.batch, c.dim, c.dstate, seg)) {
      g_last_cuda_error = "workspace smaller than ssm_scan_fwd_workspace_size()";
      return SSM_ERR_INVALID_ARG;
    }
  } else if (algo == SSM_ALGO_AUTO) {
    if (c.batch * c.dim >= kChannelKernelMinChannels) {
      algo = SSM_ALGO_CHANNEL;
    } else {
      // few channels: split a long sequence across CTAs when the caller's workspace
      // holds the segments' states; else lanes over positions (measured on B300: the
      // 130M-like layer, 3072 channels x 2048 fp32, runs 179 us over positions and
      // 306 us in 8 segments; a 1536-channel x 131072 bf16 scan 3.7 ms over positions
      // and 1.7 ms in 37 segments)
      if (c.seqlen >= kSegMinSeqlen) seg = seg_plan(c.batch, c.dim, c.seqlen, lc, false);
      algo = (seg.nseg > 1 &&
              workspace_bytes >= seg_workspace_bytes(c.batch, c.dim, c.dstate, seg))
                 ? SSM_ALGO_SEGMENTED
                 : SSM_ALGO_CHUNK;
    }
  }
  if (algo != SSM_ALGO_CHUNK && !tma_eligible(c)) algo = SSM_ALGO_CHUNK;  // TMA kernels only
  // the channel kernel with the split chosen per size: one split for every CTA, or
  // (dstate 16) the mixed launch when its model cost is lower and the workspace
  // holds its scheduler counters
  MixPlan mix;
  if (algo == SSM_ALGO_CHANNEL_MIXED) {
    mix = mix_plan(c.batch, c.dim);
    if (c.dstate != 16 || !mix.use) {
      algo = SSM_ALGO_CHANNEL;
    } else if (workspace_bytes < kStatusBytes + kMixCounterBytes) {
      g_last_cuda_error = "workspace smaller than ssm_scan_fwd_algo_workspace_size()";
      return SSM_ERR_INVALID_ARG;
    }
  } else if (algo == SSM_ALGO_CHANNEL && c.dstate == 16 &&
             workspace_bytes >= kStatusBytes + kMixCounterBytes) {
    double split_cost = 0.0;
    choose_lpc(c.batch, c.dim, c.dstate, &split_cost);
    const MixPlan m = mix_plan(c.batch, c.dim);
    if (m.use && m.k >= 1 && m.n_quarters > 0 && mix_cost(m) < split_cost) {
      mix = m;
      algo = SSM_ALGO_CHANNEL_MIXED;
    }
  }

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(ssm::DeviceStatus), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace status)");
  return c.bf16 ? dispatch_scan<uint16_t>(c, algo, workspace, s, seg, mix)
                : dispatch_scan<float>(c, algo, workspace, s, seg, mix);
}

ssm_status ssm_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ssm_dtype io,
                        const void* u, const void* delta, const float* delta_bias,
                        int delta_softplus, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* h0, float* h_last, void* y,
                        void* workspace, size_t workspace_bytes, ssm_stream_t stream) {
  return ssm_scan_fwd_algo(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A,
                           B, C, D, z, h0, h_last, y, workspace, workspace_bytes, SSM_ALGO_AUTO,
                           stream);
}

ssm_status ssm_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                ssm_dtype io, const void* u, const void* delta,
                                const float* delta_bias, int delta_softplus, const float* A,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* h0, float* h_last, void* y, ssm_stream_t stream) {
  // every plan needs the status words; the segmented long-sequence plan needs more
  // and is then skipped by AUTO (it picks the kernels whose scratch fits)
  const size_t need = kWorkspaceBytes;
  if (need > kNoAllocScratchBytes) {
    g_last_cuda_error = "ssm_scan_fwd_noalloc: these sizes need " + std::to_string(need) +
                        " bytes of scratch, more than the " +
                        std::to_string(kNoAllocScratchBytes) + " bytes reserved statically";
    return SSM_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const ssm_status st = noalloc_scratch(&scratch);
  if (st != SSM_OK) return st;
  return ssm_scan_fwd_algo(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A,
                           B, C, D, z, h0, h_last, y, scratch, kNoAllocScratchBytes, SSM_ALGO_AUTO,
                           stream);
}

ssm_status ssm_state_update(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io, float* h,
                            const void* u, const void* delta, const float* delta_bias,
                            int delta_softplus, const float* A, const void* B, const void* C,
                            const float* D, const void* z, void* y, ssm_stream_t stream) {
  ssm_status st = validate_common(batch, dim, dstate, io);
  if (st != SSM_OK) return st;
  if (batch > (int64_t(1) << 40) / dim) return SSM_ERR_INVALID_ARG;
  if (!h || !u || !delta || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
  const size_t esz = (io == SSM_DTYPE_BF16) ? 2 : 4;
  const void* io_ptrs[6] = {u, delta, B, C, y, z};
  for (const void* q : io_ptrs)
    if (q && !aligned(q, esz)) return SSM_ERR_INVALID_ARG;
  const float* f_ptrs[4] = {h, A, D, delta_bias};
  for (const float* q : f_ptrs)
    if (q && !aligned(q, 4)) return SSM_ERR_INVALID_ARG;
  UpdateParams p;
  p.batch = batch;
  p.b0 = 0;
  p.dim = static_cast<int>(dim);
  p.softplus = delta_softplus ? 1 : 0;
  p.h = h;
  p.A = A;
  p.D = D;
  p.bias = delta_bias;
  p.u = u;
  p.delta = delta;
  p.z = z;
  p.B = B;
  p.C = C;
  p.y = y;
  // 16-byte vectors for h and A, 4-element vectors for B and C
  const bool vec = aligned(h, 16) && aligned(A, 16) && aligned(B, 4 * esz) && aligned(C, 4 * esz);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return (io == SSM_DTYPE_BF16) ? dispatch_update<uint16_t>(p, dstate, vec, s)
                                : dispatch_update<float>(p, dstate, vec, s);
}

ssm_status ssm_read_device_status(const void* workspace, ssm_stream_t stream) {
  if (!workspace || !aligned(workspace, 16)) return SSM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  ssm::DeviceStatus st;
  e = cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(workspace status)");
  return (st.flags & ssm::kStatusTimeout) ? SSM_ERR_DEVICE_TIMEOUT : SSM_OK;
}

const char* ssm_status_string(ssm_status status) {
  switch (status) {
    case SSM_OK: return "SSM_OK: success";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG: invalid size, NULL or misaligned pointer";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: dstate, dtype or algorithm not supported";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA: a CUDA call or kernel launch failed";
    case SSM_ERR_DEVICE_TIMEOUT: return "SSM_ERR_DEVICE_TIMEOUT: a device-side wait hit its limit";
  }
  return "unknown ssm_status";
}

const char* ssm_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int ssm_version(void) { return kVersion; }

}  // extern "C"
