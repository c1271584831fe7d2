// ssm_host.cuh -- host-side pieces shared by the translation units of libssm:
// argument checks, TMA descriptor encoding, plan choice (lane split, mixed split,
// segments) and the declarations of the per-type dispatchers that the kernel
// translation units define and instantiate.
#pragma once

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
#include "conv1d.cuh"
#include "scan_bwd.cuh"

namespace ssm_host {

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

inline thread_local std::string g_last_cuda_error;
inline thread_local std::string g_last_plan;

inline ssm_status cuda_fail(cudaError_t e, const char* what) {
  g_last_cuda_error = std::string(what) + ": " + cudaGetErrorString(e);
  return SSM_ERR_CUDA;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// TMA descriptor encoding through the driver entry point
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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
inline bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
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
  float* ckpt = nullptr;  // training forward: state checkpoints (else null)
  // where the kernels record wait timeouts (null: the first bytes of the workspace)
  ssm::DeviceStatus* status = nullptr;
  int softplus;
  bool euler;  // input term dt * B instead of the ZOH form
};

inline ssm_status validate_common(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io) {
  if (batch < 1 || dim < 1 || dstate < 1) return SSM_ERR_INVALID_ARG;
  if (io != SSM_DTYPE_F32 && io != SSM_DTYPE_BF16) return SSM_ERR_UNSUPPORTED;
  if (dstate != 4 && dstate != 8 && dstate != 16) return SSM_ERR_UNSUPPORTED;
  if (dim > INT32_MAX || batch > INT32_MAX) return SSM_ERR_INVALID_ARG;
  return SSM_OK;
}

inline ssm_status validate_scan(const ScanCall& c, const void* workspace, size_t workspace_bytes) {
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

inline bool tma_eligible(const ScanCall& c) {
  const int64_t esz = c.bf16 ? 2 : 4;
  if ((c.seqlen * esz) % 16 != 0) return false;
  const void* ptrs[6] = {c.u, c.delta, c.B, c.C, c.y, c.z};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return false;
  return encode_fn() != nullptr;
}

inline bool vec_eligible(const ScanCall& c) {
  const int64_t esz = c.bf16 ? 2 : 4;
  if ((c.seqlen * esz) % 16 != 0) return false;
  const void* ptrs[6] = {c.u, c.delta, c.B, c.C, c.y, c.z};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return false;
  return true;
}

// SM count of the current device (cached per device ordinal).
inline int sm_count() {
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

inline ScanParams make_params(const ScanCall& c, void* workspace) {
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
  p.status = c.status ? c.status : static_cast<ssm::DeviceStatus*>(workspace);
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
  p.ckpt = c.ckpt;
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

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SegPlan {
  int nseg = 1;     // 1: not segmented
  int seg_len = 0;
};

// Segments for the one-lane-per-channel channel kernel: enough that the CTAs fill
// every SM (kSegCtasPerSm per SM), each at least kSegMinLen positions long, a
// multiple of the chunk (lc positions).  `force` asks for at least two segments.
inline SegPlan seg_plan(int64_t batch, int64_t dim, int64_t seqlen, int lc, bool force) {
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

inline size_t seg_workspace_bytes(int64_t batch, int64_t dim, int64_t dstate, const SegPlan& pl) {
  if (pl.nseg < 2) return kStatusBytes;
  const size_t chans = static_cast<size_t>(batch) * static_cast<size_t>(dim);
  return kStatusBytes + round_up(static_cast<size_t>(pl.nseg) * chans * dstate * 4, 256) +
         round_up(static_cast<size_t>(pl.nseg) * chans * 4, 256);
}

// bytes of the training forward's state checkpoints: the state entering every block of
// ssm::kCkptPos positions, [ceil(seqlen / kCkptPos)][batch * dim][dstate] fp32
inline size_t ckpt_bytes(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
  return static_cast<size_t>((seqlen + ssm::kCkptPos - 1) / ssm::kCkptPos) *
         static_cast<size_t>(batch) * static_cast<size_t>(dim) * static_cast<size_t>(dstate) * 4;
}

// ---------------------------------------------------------------------------
// scan gradient workspace: [0, 256) status words; the block checkpoints
// [nblk][batch * dim][N]; the per-CTA dB / dC partials [tiles][batch][2][N][L];
// the per-(segment, channel) dA [nseg][batch * dim][N], dD and bias gradient
// [nseg][batch * dim][2]; with segments, their end states and own adjoints
// [nseg][batch * dim][N] each and step-size sums [nseg][batch * dim]; one byte per
// CTA [nseg][batch][tiles] saying whether it takes the fast coefficients
// ---------------------------------------------------------------------------
constexpr int kBwdThreads = 128;
static_assert(ssm::kBwdPos == ssm::kCkptPos,
              "the gradient's blocks are the training forward's checkpoint blocks");
constexpr int kBwdChannels = kBwdThreads / ssm::kBwdLpc;
// split sequences until about this many (segment, tile) CTAs per SM: four waves of
// the four resident CTAs (measured on the long-sequence gradient, B1 D1536 L131072:
// 13 segments 12.8 ms, 26 10.8 ms, 52 9.9 ms, 78 9.7 ms; unsplit 48.8 ms)
constexpr int kBwdSegCtasPerSm = 16;
constexpr int64_t kBwdMinSegLen = 256;   // positions: shorter segments cost more than they gain

struct BwdLayout {
  int64_t nblk = 0, tiles = 0;
  int nseg = 1, seg_len = 0;
  size_t off_ckpt = 0, off_bc = 0, off_a = 0, off_dd = 0, off_E = 0, off_R = 0, off_sum = 0,
         off_flags = 0, total = 0;
};

// Segments for the gradient: when the (batch row, channel tile) CTAs cannot fill
// the SMs (fewer than two per SM), split the sequence into about
// kBwdSegCtasPerSm CTAs per SM, each segment at least kBwdMinSegLen positions, a
// multiple of the 8-position block.  `segments` > 0 asks for that many (tests).
// `own_ckpt`: the workspace holds the checkpoints (false when the training forward's
// are given)
inline BwdLayout bwd_layout(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                            int64_t segments = 0, bool own_ckpt = true) {
  BwdLayout w;
  w.nblk = (seqlen + ssm::kBwdPos - 1) / ssm::kBwdPos;
  w.tiles = (dim + kBwdChannels - 1) / kBwdChannels;
  const int64_t ctas = batch * w.tiles;
  int64_t nseg = 1;
  if (segments > 0) {
    nseg = segments;
  } else if (ctas < 2 * static_cast<int64_t>(sm_count())) {
    nseg = (static_cast<int64_t>(sm_count()) * kBwdSegCtasPerSm + ctas - 1) / ctas;
    if (nseg > seqlen / kBwdMinSegLen) nseg = seqlen / kBwdMinSegLen;
  }
  if (nseg > w.nblk) nseg = w.nblk;
  if (nseg < 1) nseg = 1;
  int64_t len = (seqlen + nseg - 1) / nseg;
  len = (len + ssm::kBwdPos - 1) / ssm::kBwdPos * ssm::kBwdPos;
  w.nseg = static_cast<int>((seqlen + len - 1) / len);
  w.seg_len = static_cast<int>(w.nseg == 1 ? seqlen : len);
  const size_t rows = static_cast<size_t>(batch) * static_cast<size_t>(dim);
  const size_t ns = static_cast<size_t>(w.nseg);
  w.off_ckpt = kStatusBytes;
  w.off_bc = w.off_ckpt +
             (own_ckpt ? round_up(static_cast<size_t>(w.nblk) * rows * dstate * 4, 256) : 0);
  w.off_a = w.off_bc + round_up(static_cast<size_t>(w.tiles) * batch * 2 * dstate *
                                    static_cast<size_t>(seqlen) * 4, 256);
  w.off_dd = w.off_a + round_up(ns * rows * dstate * 4, 256);
  w.off_E = w.off_dd + round_up(ns * rows * 2 * 4, 256);
  if (w.nseg > 1) {
    w.off_R = w.off_E + round_up(ns * rows * dstate * 4, 256);
    w.off_sum = w.off_R + round_up(ns * rows * dstate * 4, 256);
    w.off_flags = w.off_sum + round_up(ns * rows * 4, 256);
  } else {
    w.off_R = w.off_sum = w.off_E;
    w.off_flags = w.off_E;
  }
  // one byte per CTA: fast or accurate coefficients
  w.total = w.off_flags + round_up(ns * static_cast<size_t>(batch) * w.tiles, 256);
  return w;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Channel-kernel shapes: 64-byte chunk rows (32 bf16 / 16 fp32 positions) in a
// 2-stage ring.  A CTA meets its warps at a barrier once per chunk: 64-byte rows
// halve those meetings against 32-byte ones (measured on B300, one-lane CTAs of
// the 2.8B-like layer's arithmetic at 2 warps per SM sub-partition: 481 -> 446 us),
// and two stages of them keep as many positions in flight as four of 32 bytes.
// Per 4-warp CTA (bf16, dstate 16, gate): ~61 KB of shared memory at 1 lane per
// channel (3 CTAs per SM), less at 2 and 4.
template <int LPC>
struct ChanShape {
  static constexpr int S = 2, RB = 64;
};

// Lanes per channel for the channel kernel.  Every SM sub-partition runs one warp
// of each resident CTA, so the busiest sub-partition processes kmax = ceil(CTAs /
// SMs) warps.  Its time is the larger of kmax x the issue cost of one warp (which
// falls with the states a lane holds, NS = dstate / LPC, but less than in
// proportion because the per-position work and the lane exchange do not shrink)
// and the latency of a single warp when there are too few warps to overlap.  The
// relative costs below were measured on B300 with the 2.8B-like layer (bf16,
// dstate 16, L 2048): one warp of NS = 16 / 8 / 4 states costs 1 / 0.58 / 0.37
// when sub-partitions are full, and a lone warp takes 1.78 / 1.6 / 1.2.
inline int choose_lpc(int64_t batch, int64_t dim, int64_t dstate, double* cost_out = nullptr) {
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

inline MixPlan mix_plan(int64_t batch, int64_t dim) {
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

inline double mix_cost(const MixPlan& m) {
  const int64_t sms = sm_count();
  return m.k * 1.0 + double((m.n_quarters + sms - 1) / sms) * 0.37;
}


// Launch one kernel family for element type IO, dstate N and input term EULER
// (defined in ssm_launch.cuh, instantiated in the inst_*.cu translation units).
template <typename IO, int N, bool EULER>
ssm_status dispatch_scan_n(const ScanCall& c, ssm_algo algo, void* ws, cudaStream_t s,
                           const SegPlan& seg, const MixPlan& mix);
template <typename IO, int N, bool EULER>
ssm_status dispatch_update_n(const ssm::UpdateParams& p, bool vec, cudaStream_t s);

// Causal conv1d launches (defined in inst_conv.cu).  `vec`: x, out 16-byte aligned
// and rows a multiple of 16 bytes long.
ssm_status launch_conv1d_fwd(bool bf16, const ssm::ConvParams& p, bool vec, cudaStream_t s);
// scan gradient: the main kernel and the two reductions (inst_bwd_*.cu)
template <typename IO>
ssm_status launch_scan_bwd(const ssm::BwdParams& p, int dstate, bool gate, bool euler, bool vec,
                           void* dB, void* dC, float* dA, float* dD, float* dbias,
                           cudaStream_t s);
ssm_status launch_conv1d_update(bool bf16, const ssm::ConvParams& p, cudaStream_t s);

}  // namespace ssm_host
