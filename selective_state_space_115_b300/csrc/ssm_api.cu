// ssm_api.cu -- C ABI of libssm (declared in include/ssm.h).
//
// Host side: argument validation (nothing is enqueued when it fails), choice of
// kernel family, TMA descriptor encoding, launches on the caller's stream.
// The library allocates no device memory and keeps no per-call state (except the
// statically reserved scratch of ssm_scan_fwd_noalloc, below).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "ssm.h"
#include "ssm_host.cuh"

namespace {

using namespace ssm_host;

template <typename IO>
ssm_status dispatch_scan(const ScanCall& c, ssm_algo algo, void* ws, cudaStream_t s,
                         const SegPlan& seg, const MixPlan& mix) {
  switch (c.dstate) {
    case 4:
      return c.euler ? dispatch_scan_n<IO, 4, true>(c, algo, ws, s, seg, mix)
                     : dispatch_scan_n<IO, 4, false>(c, algo, ws, s, seg, mix);
    case 8:
      return c.euler ? dispatch_scan_n<IO, 8, true>(c, algo, ws, s, seg, mix)
                     : dispatch_scan_n<IO, 8, false>(c, algo, ws, s, seg, mix);
    case 16:
      return c.euler ? dispatch_scan_n<IO, 16, true>(c, algo, ws, s, seg, mix)
                     : dispatch_scan_n<IO, 16, false>(c, algo, ws, s, seg, mix);
    default: return SSM_ERR_UNSUPPORTED;
  }
}

template <typename IO>
ssm_status dispatch_update(const UpdateParams& p, int64_t dstate, bool vec, bool euler,
                           cudaStream_t s) {
  switch (dstate) {
    case 4: return euler ? dispatch_update_n<IO, 4, true>(p, vec, s)
                         : dispatch_update_n<IO, 4, false>(p, vec, s);
    case 8: return euler ? dispatch_update_n<IO, 8, true>(p, vec, s)
                         : dispatch_update_n<IO, 8, false>(p, vec, s);
    case 16: return euler ? dispatch_update_n<IO, 16, true>(p, vec, s)
                          : dispatch_update_n<IO, 16, false>(p, vec, s);
    default: return SSM_ERR_UNSUPPORTED;
  }
}

// ---------------------------------------------------------------------------
// statically reserved scratch for ssm_scan_fwd_noalloc
// ---------------------------------------------------------------------------
// Device scratch of fixed size that every GPU loading this library holds until
// the process exits.  Host code must not pass the symbol itself to a kernel (on
// the host it only names a stand-in object); the device address is looked up with
// cudaGetSymbolAddress for the current device's context.  The address belongs to
// that context: after cudaDeviceReset (or the primary context being released and
// created again) the module loads anew and the array may move, so the cached
// address is keyed by the context's unique id and looked up again when it changes.
constexpr size_t kNoAllocScratchBytes = 4096;
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
struct NoAllocSlot {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
NoAllocSlot g_noalloc[kNoAllocMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// unique id of the calling thread's current context (0 when it cannot be read: the
// address is then looked up on every call)
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = []() -> CtxGetCurrentFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  static CtxGetIdFn get_id = []() -> CtxGetIdFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetIdFn>(f);
  }();
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the static scratch in the current device's context: looked up
// on the first call in a context (the runtime then makes the device's primary
// context current and loads the module if it has not yet) and kept for later calls
// in the same context.
ssm_status noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    g_last_cuda_error = "ssm_scan_fwd_noalloc: device ordinal beyond the supported range";
    return SSM_ERR_UNSUPPORTED;
  }
  // nothing cached yet: look up first (that call also makes the primary context
  // current), then record the context it belongs to
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocSlot& slot = g_noalloc[dev];
  unsigned long long id = slot.ptr ? current_context_id() : 0;
  if (!slot.ptr || id == 0 || id != slot.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    slot.ptr = p;
    slot.ctx_id = current_context_id();
  }
  *out = slot.ptr;
  return SSM_OK;
}

// Text of the plan a scan-forward call launched (for ssm_last_plan).
std::string describe_plan(const ScanCall& c, ssm_algo algo, const SegPlan& seg,
                          const MixPlan& mix) {
  const std::string io = c.bf16 ? "bf16" : "fp32";
  const std::string n = std::to_string(c.dstate);
  switch (algo) {
    case SSM_ALGO_CHANNEL_MIXED:
      return "scan_channel_mixed_kernel<" + io + ", N" + n + ">: " + std::to_string(mix.k) +
             " one-lane-per-channel CTAs of 128 channels per SM (" +
             std::to_string(mix.n_tiles) + ") + " + std::to_string(mix.n_quarters) +
             " four-lane CTAs of 32 channels";
    case SSM_ALGO_SEGMENTED:
      return "scan_channel_kernel<" + io + ", N" + n + "> segmented: " +
             std::to_string(seg.nseg) + " segments of " + std::to_string(seg.seg_len) +
             " positions, pass 1 (segment end states) + pass 2 (outputs)";
    case SSM_ALGO_CHANNEL:
      return "scan_channel_kernel<" + io + ", N" + n + ">: " +
             std::to_string(choose_lpc(c.batch, c.dim, c.dstate)) + " lane(s) per channel";
    case SSM_ALGO_CHANNEL_L1: return "scan_channel_kernel<" + io + ", N" + n + ">: 1 lane per channel";
    case SSM_ALGO_CHANNEL_L2: return "scan_channel_kernel<" + io + ", N" + n + ">: 2 lanes per channel";
    case SSM_ALGO_CHANNEL_L4: return "scan_channel_kernel<" + io + ", N" + n + ">: 4 lanes per channel";
    default:
      return "scan_chunk_kernel<" + io + ", N" + n + ">: one warp per channel, lanes over positions";
  }
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

}  // extern "C"

namespace {

// AUTO's plan for a call: the channel kernel for many channels; for few, a long
// sequence split across CTAs when `workspace_bytes` holds the segments' states, else
// lanes over positions (measured on B300: the 130M-like layer, 3072 channels x 2048
// fp32, runs 179 us over positions and 306 us in 8 segments; a 1536-channel x 131072
// bf16 scan 3.7 ms over positions and 1.7 ms in 37 segments).
ssm_algo auto_plan(const ScanCall& c, size_t workspace_bytes, int lc, SegPlan* seg) {
  if (c.batch * c.dim >= kChannelKernelMinChannels) return SSM_ALGO_CHANNEL;
  if (c.seqlen >= kSegMinSeqlen) *seg = seg_plan(c.batch, c.dim, c.seqlen, lc, false);
  return (seg->nseg > 1 && workspace_bytes >= seg_workspace_bytes(c.batch, c.dim, c.dstate, *seg))
             ? SSM_ALGO_SEGMENTED
             : SSM_ALGO_CHUNK;
}

// The channel kernel with the split chosen per size becomes the mixed launch (dstate
// 16) when its model cost is lower and the workspace holds its scheduler counters.
ssm_algo mixed_upgrade(const ScanCall& c, size_t workspace_bytes, MixPlan* mix) {
  if (c.dstate != 16 || workspace_bytes < kStatusBytes + kMixCounterBytes)
    return SSM_ALGO_CHANNEL;
  double split_cost = 0.0;
  choose_lpc(c.batch, c.dim, c.dstate, &split_cost);
  const MixPlan m = mix_plan(c.batch, c.dim);
  if (m.use && m.k >= 1 && m.n_quarters > 0 && mix_cost(m) < split_cost) {
    *mix = m;
    return SSM_ALGO_CHANNEL_MIXED;
  }
  return SSM_ALGO_CHANNEL;
}

// The scan forward; `ckpt` (training forward) receives the state checkpoints, else null.
ssm_status scan_fwd_impl(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                         ssm_dtype io, const void* u, const void* delta, const float* delta_bias,
                         int delta_softplus, const float* A, const void* B, const void* C,
                         const float* D, const void* z, const float* h0, float* h_last, void* y,
                         float* ckpt, void* workspace, size_t workspace_bytes,
                         ssm_discretization disc, ssm_algo algo, ssm_stream_t stream) {
  if (disc != SSM_DISC_ZOH && disc != SSM_DISC_EULER) return SSM_ERR_UNSUPPORTED;
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
  c.euler = (disc == SSM_DISC_EULER);
  c.ckpt = ckpt;
  if (io != SSM_DTYPE_F32 && io != SSM_DTYPE_BF16) return SSM_ERR_UNSUPPORTED;
  ssm_status st = validate_scan(c, workspace, workspace_bytes);
  if (st != SSM_OK) return st;

  const int lc = ChanShape<1>::RB / (c.bf16 ? 2 : 4);  // channel kernel chunk (positions)
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
    algo = auto_plan(c, workspace_bytes, lc, &seg);
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
  } else if (algo == SSM_ALGO_CHANNEL) {
    algo = mixed_upgrade(c, workspace_bytes, &mix);
  }

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(ssm::DeviceStatus), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace status)");
  const ssm_status rs = c.bf16 ? dispatch_scan<uint16_t>(c, algo, workspace, s, seg, mix)
                               : dispatch_scan<float>(c, algo, workspace, s, seg, mix);
  if (rs == SSM_OK) g_last_plan = describe_plan(c, algo, seg, mix);
  return rs;
}

// The gradient's own forward pass on the forward's kernels: the state entering every
// kCkptPos positions into `ckpt`, no output (neither C nor z read).  It takes AUTO's
// plan when that is the channel kernel (one split, the mixed launch or segments) and
// returns SSM_ERR_UNSUPPORTED otherwise, where the gradient then forms its checkpoints
// itself.  `scratch` holds the plan's scheduler counters or segment states; wait
// timeouts go to `status`.
ssm_status ckpt_forward(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, bool bf16,
                        const void* u, const void* delta, const float* delta_bias, int softplus,
                        const float* A, const void* B, const void* C, const float* h0, bool euler,
                        float* ckpt, void* scratch, size_t scratch_bytes,
                        ssm::DeviceStatus* status, cudaStream_t s) {
  ScanCall c;
  c.batch = batch;
  c.dim = dim;
  c.dstate = dstate;
  c.seqlen = seqlen;
  c.bf16 = bf16;
  c.u = u;
  c.delta = delta;
  c.B = B;
  c.C = C;
  c.z = nullptr;
  c.bias = delta_bias;
  c.A = A;
  c.D = nullptr;
  c.h0 = h0;
  c.h_last = nullptr;
  c.y = nullptr;
  c.ckpt = ckpt;
  c.status = status;
  c.softplus = softplus ? 1 : 0;
  c.euler = euler;
  if (!tma_eligible(c) || (c.batch * c.dim + 3) / 4 > INT32_MAX) return SSM_ERR_UNSUPPORTED;
  const int lc = ChanShape<1>::RB / (c.bf16 ? 2 : 4);
  SegPlan seg;
  MixPlan mix;
  ssm_algo algo = auto_plan(c, scratch_bytes, lc, &seg);
  if (algo == SSM_ALGO_CHUNK) return SSM_ERR_UNSUPPORTED;
  if (algo == SSM_ALGO_CHANNEL) algo = mixed_upgrade(c, scratch_bytes, &mix);
  const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(ssm::DeviceStatus), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  return c.bf16 ? dispatch_scan<uint16_t>(c, algo, scratch, s, seg, mix)
                : dispatch_scan<float>(c, algo, scratch, s, seg, mix);
}

}  // namespace

extern "C" {

ssm_status ssm_scan_fwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                           ssm_dtype io, const void* u, const void* delta, const float* delta_bias,
                           int delta_softplus, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* h0, float* h_last,
                           void* y, void* workspace, size_t workspace_bytes,
                           ssm_discretization disc, ssm_algo algo, ssm_stream_t stream) {
  return scan_fwd_impl(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A, B,
                       C, D, z, h0, h_last, y, nullptr, workspace, workspace_bytes, disc, algo,
                       stream);
}

size_t ssm_scan_ckpt_bytes(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1) return 0;
  if (batch > (int64_t(1) << 62) / dim / seqlen / dstate) return 0;
  return ckpt_bytes(batch, dim, dstate, seqlen);
}

ssm_status ssm_scan_fwd_train(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                              ssm_dtype io, const void* u, const void* delta,
                              const float* delta_bias, int delta_softplus, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              const float* h0, float* h_last, void* y, float* ckpt,
                              size_t ckpt_bytes_given, void* workspace, size_t workspace_bytes,
                              ssm_discretization disc, ssm_algo algo, ssm_stream_t stream) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1) return SSM_ERR_INVALID_ARG;
  if (batch > (int64_t(1) << 62) / dim / seqlen / dstate) return SSM_ERR_INVALID_ARG;
  if (!ckpt || !aligned(ckpt, 16)) return SSM_ERR_INVALID_ARG;
  if (ckpt_bytes_given < ckpt_bytes(batch, dim, dstate, seqlen)) {
    g_last_cuda_error = "checkpoint buffer smaller than ssm_scan_ckpt_bytes()";
    return SSM_ERR_INVALID_ARG;
  }
  return scan_fwd_impl(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A, B,
                       C, D, z, h0, h_last, y, ckpt, workspace, workspace_bytes, disc, algo,
                       stream);
}

ssm_status ssm_scan_fwd_algo(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             ssm_dtype io, const void* u, const void* delta,
                             const float* delta_bias, int delta_softplus, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* h0, float* h_last, void* y, void* workspace,
                             size_t workspace_bytes, ssm_algo algo, ssm_stream_t stream) {
  return ssm_scan_fwd_ex(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A,
                         B, C, D, z, h0, h_last, y, workspace, workspace_bytes, SSM_DISC_ZOH, algo,
                         stream);
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
  // AUTO picks among the plans whose scratch fits the reserved bytes: the status
  // words and the mixed split's counters always do; the segmented long-sequence plan
  // when its segment states fit, else the lanes-over-positions kernel takes its place
  static_assert(kStatusBytes + kMixCounterBytes <= kNoAllocScratchBytes,
                "the channel kernels' scratch fits the reserved array");
  void* scratch = nullptr;
  const ssm_status st = noalloc_scratch(&scratch);
  if (st != SSM_OK) return st;
  return ssm_scan_fwd_algo(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A,
                           B, C, D, z, h0, h_last, y, scratch, kNoAllocScratchBytes, SSM_ALGO_AUTO,
                           stream);
}

ssm_status ssm_state_update_ex(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io,
                               float* h, const void* u, const void* delta,
                               const float* delta_bias, int delta_softplus, const float* A,
                               const void* B, const void* C, const float* D, const void* z,
                               void* y, ssm_discretization disc, ssm_stream_t stream) {
  if (disc != SSM_DISC_ZOH && disc != SSM_DISC_EULER) return SSM_ERR_UNSUPPORTED;
  const bool euler = (disc == SSM_DISC_EULER);
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
  return (io == SSM_DTYPE_BF16) ? dispatch_update<uint16_t>(p, dstate, vec, euler, s)
                                : dispatch_update<float>(p, dstate, vec, euler, s);
}

ssm_status ssm_state_update(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io, float* h,
                            const void* u, const void* delta, const float* delta_bias,
                            int delta_softplus, const float* A, const void* B, const void* C,
                            const float* D, const void* z, void* y, ssm_stream_t stream) {
  return ssm_state_update_ex(batch, dim, dstate, io, h, u, delta, delta_bias, delta_softplus, A, B,
                             C, D, z, y, SSM_DISC_ZOH, stream);
}

size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
  return ssm_scan_bwd_ex_workspace_size(batch, dim, dstate, seqlen, 0);
}

size_t ssm_scan_bwd_ex_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                      int segments) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1 || segments < 0) return kStatusBytes;
  return bwd_layout(batch, dim, dstate, seqlen, segments).total;
}

ssm_status ssm_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ssm_dtype io,
                        const void* u, const void* delta, const float* delta_bias,
                        int delta_softplus, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* h0, const void* dy,
                        const float* dh_last, void* du, void* ddelta, float* dA, void* dB,
                        void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                        void* workspace, size_t workspace_bytes, ssm_discretization disc,
                        ssm_stream_t stream) {
  return ssm_scan_bwd_ex(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A,
                         B, C, D, z, h0, dy, dh_last, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                         dh0, workspace, workspace_bytes, disc, 0, stream);
}

}  // extern "C"

namespace {

// The scan gradient; `ckpt_in` (from the training forward) gives every block's entering
// state, else null (the gradient recomputes them).
ssm_status scan_bwd_impl(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                         ssm_dtype io, const void* u, const void* delta, const float* delta_bias,
                         int delta_softplus, const float* A, const void* B, const void* C,
                         const float* D, const void* z, const float* h0, const float* ckpt_in,
                         const void* dy, const float* dh_last, void* du, void* ddelta, float* dA,
                         void* dB, void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                         void* workspace, size_t workspace_bytes, ssm_discretization disc,
                         int segments, ssm_stream_t stream) {
  if (segments < 0) return SSM_ERR_INVALID_ARG;
  ssm_status st = validate_common(batch, dim, dstate, io);
  if (st != SSM_OK) return st;
  if (seqlen < 1 || seqlen > INT32_MAX - 4096) return SSM_ERR_INVALID_ARG;
  if (batch > (int64_t(1) << 62) / dim / seqlen / dstate) return SSM_ERR_INVALID_ARG;
  if (disc != SSM_DISC_ZOH && disc != SSM_DISC_EULER) return SSM_ERR_INVALID_ARG;
  if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC)
    return SSM_ERR_INVALID_ARG;
  if ((z != nullptr) != (dz != nullptr)) return SSM_ERR_INVALID_ARG;
  if (D && !dD) return SSM_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return SSM_ERR_INVALID_ARG;
  const BwdLayout w = bwd_layout(batch, dim, dstate, seqlen, segments, ckpt_in == nullptr);
  if (workspace_bytes < w.total) return SSM_ERR_INVALID_ARG;
  if (ckpt_in && !aligned(ckpt_in, 4)) return SSM_ERR_INVALID_ARG;
  const size_t esz = (io == SSM_DTYPE_BF16) ? 2 : 4;
  const void* io_ptrs[12] = {u, delta, B, C, z, dy, du, ddelta, dB, dC, dz, nullptr};
  for (const void* q : io_ptrs)
    if (q && !aligned(q, esz)) return SSM_ERR_INVALID_ARG;
  const void* f_ptrs[10] = {delta_bias, A, D, h0, dh_last, dA, dD, ddelta_bias, dh0, nullptr};
  for (const void* q : f_ptrs)
    if (q && !aligned(q, 4)) return SSM_ERR_INVALID_ARG;
  // cp.async staging and 16-byte output stores need 16-byte rows
  bool vec = (seqlen * static_cast<int64_t>(esz)) % 16 == 0;
  const void* v_ptrs[7] = {u, delta, z, dy, du, ddelta, dz};
  for (const void* q : v_ptrs)
    if (q && !aligned(q, 16)) vec = false;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  ssm::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = batch;
  p.dim = static_cast<int>(dim);
  p.seqlen = static_cast<int>(seqlen);
  p.nblk = static_cast<int>(w.nblk);
  p.tiles = static_cast<int>(w.tiles);
  p.softplus = delta_softplus ? 1 : 0;
  p.u = u;
  p.delta = delta;
  p.z = z;
  p.dy = dy;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.bias = delta_bias;
  p.h0 = h0;
  p.dh_last = dh_last;
  p.du = du;
  p.ddelta = ddelta;
  p.dz = dz;
  p.dh0 = dh0;
  p.ckpt = reinterpret_cast<float*>(ws + w.off_ckpt);
  p.part_bc = reinterpret_cast<float*>(ws + w.off_bc);
  p.part_a = reinterpret_cast<float*>(ws + w.off_a);
  p.part_dd = reinterpret_cast<float*>(ws + w.off_dd);
  p.nseg = w.nseg;
  p.seg_len = w.seg_len;
  p.seg_E = reinterpret_cast<float*>(ws + w.off_E);
  p.seg_R = reinterpret_cast<float*>(ws + w.off_R);
  p.seg_sum = reinterpret_cast<float*>(ws + w.off_sum);
  p.cta_fast = ws + w.off_flags;
  p.ckpt_in = ckpt_in;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!ckpt_in && segments == 0) {
    // the checkpoints from the forward's channel kernels (cheaper per update than the
    // gradient kernel's own forward pass), in the workspace's checkpoint region; the
    // dB/dC partials' region, unused until the gradient kernel, is their scratch, and
    // the workspace's first bytes their status words
    const ssm_status fs = ckpt_forward(
        batch, dim, dstate, seqlen, io == SSM_DTYPE_BF16, u, delta, delta_bias, delta_softplus,
        A, B, C, h0, disc == SSM_DISC_EULER, p.ckpt, ws + w.off_bc, w.off_a - w.off_bc,
        reinterpret_cast<ssm::DeviceStatus*>(ws), s);
    if (fs == SSM_OK) {
      p.ckpt_in = p.ckpt;
    } else if (fs != SSM_ERR_UNSUPPORTED) {
      return fs;
    }
  }
  const bool euler = disc == SSM_DISC_EULER;
  float* dD_out = D ? dD : nullptr;
  if (io == SSM_DTYPE_BF16)
    return launch_scan_bwd<uint16_t>(p, static_cast<int>(dstate), z != nullptr, euler, vec, dB,
                                     dC, dA, dD_out, ddelta_bias, s);
  return launch_scan_bwd<float>(p, static_cast<int>(dstate), z != nullptr, euler, vec, dB, dC, dA,
                                dD_out, ddelta_bias, s);
}

}  // namespace

extern "C" {

ssm_status ssm_scan_bwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                           ssm_dtype io, const void* u, const void* delta, const float* delta_bias,
                           int delta_softplus, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* h0, const void* dy,
                           const float* dh_last, void* du, void* ddelta, float* dA, void* dB,
                           void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                           void* workspace, size_t workspace_bytes, ssm_discretization disc,
                           int segments, ssm_stream_t stream) {
  return scan_bwd_impl(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A, B,
                       C, D, z, h0, nullptr, dy, dh_last, du, ddelta, dA, dB, dC, dD, dz,
                       ddelta_bias, dh0, workspace, workspace_bytes, disc, segments, stream);
}

size_t ssm_scan_bwd_ckpt_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                        int64_t seqlen, int segments) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1 || segments < 0) return kStatusBytes;
  return bwd_layout(batch, dim, dstate, seqlen, segments, false).total;
}

ssm_status ssm_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             ssm_dtype io, const void* u, const void* delta,
                             const float* delta_bias, int delta_softplus, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* h0, const float* ckpt, const void* dy,
                             const float* dh_last, void* du, void* ddelta, float* dA, void* dB,
                             void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                             void* workspace, size_t workspace_bytes, ssm_discretization disc,
                             int segments, ssm_stream_t stream) {
  if (!ckpt) return SSM_ERR_INVALID_ARG;
  return scan_bwd_impl(batch, dim, dstate, seqlen, io, u, delta, delta_bias, delta_softplus, A, B,
                       C, D, z, h0, ckpt, dy, dh_last, du, ddelta, dA, dB, dC, dD, dz,
                       ddelta_bias, dh0, workspace, workspace_bytes, disc, segments, stream);
}

ssm_status ssm_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                          ssm_dtype io, const void* x, const float* weight, const float* bias,
                          const void* conv_state, int apply_silu, void* out,
                          void* conv_state_out, ssm_stream_t stream) {
  ssm_status st = validate_common(batch, dim, 4, io);
  if (st != SSM_OK) return st;
  if (seqlen < 1 || seqlen > INT32_MAX - 16) return SSM_ERR_INVALID_ARG;
  if (width < 1 || width > ssm::kConvMaxWidth) return SSM_ERR_UNSUPPORTED;
  if (batch > (int64_t(1) << 62) / dim / seqlen) return SSM_ERR_INVALID_ARG;
  if (!x || !weight || !out) return SSM_ERR_INVALID_ARG;
  const size_t esz = (io == SSM_DTYPE_BF16) ? 2 : 4;
  const void* io_ptrs[4] = {x, out, conv_state, conv_state_out};
  for (const void* q : io_ptrs)
    if (q && !aligned(q, esz)) return SSM_ERR_INVALID_ARG;
  if (!aligned(weight, 4) || (bias && !aligned(bias, 4))) return SSM_ERR_INVALID_ARG;
  ssm::ConvParams p;
  std::memset(&p, 0, sizeof(p));
  p.rows = batch * dim;
  p.dim = static_cast<int>(dim);
  p.seqlen = static_cast<int>(seqlen);
  p.width = static_cast<int>(width);
  p.silu = apply_silu ? 1 : 0;
  p.x = x;
  p.w = weight;
  p.bias = bias;
  p.state_in = conv_state;
  p.out = out;
  p.state_out = conv_state_out;
  const bool vec = (seqlen * static_cast<int64_t>(esz)) % 16 == 0 && aligned(x, 16) &&
                   aligned(out, 16);
  return launch_conv1d_fwd(io == SSM_DTYPE_BF16, p, vec, reinterpret_cast<cudaStream_t>(stream));
}

ssm_status ssm_conv1d_update(int64_t batch, int64_t dim, int64_t width, ssm_dtype io,
                             void* conv_state, const void* x, const float* weight,
                             const float* bias, int apply_silu, void* out, ssm_stream_t stream) {
  ssm_status st = validate_common(batch, dim, 4, io);
  if (st != SSM_OK) return st;
  if (width < 1 || width > ssm::kConvMaxWidth) return SSM_ERR_UNSUPPORTED;
  if (batch > (int64_t(1) << 40) / dim) return SSM_ERR_INVALID_ARG;
  if (!x || !weight || !out || (width > 1 && !conv_state)) return SSM_ERR_INVALID_ARG;
  const size_t esz = (io == SSM_DTYPE_BF16) ? 2 : 4;
  const void* io_ptrs[3] = {x, out, conv_state};
  for (const void* q : io_ptrs)
    if (q && !aligned(q, esz)) return SSM_ERR_INVALID_ARG;
  if (!aligned(weight, 4) || (bias && !aligned(bias, 4))) return SSM_ERR_INVALID_ARG;
  ssm::ConvParams p;
  std::memset(&p, 0, sizeof(p));
  p.rows = batch * dim;
  p.dim = static_cast<int>(dim);
  p.width = static_cast<int>(width);
  p.silu = apply_silu ? 1 : 0;
  p.x = x;
  p.w = weight;
  p.bias = bias;
  p.out = out;
  p.state = conv_state;
  return launch_conv1d_update(io == SSM_DTYPE_BF16, p, reinterpret_cast<cudaStream_t>(stream));
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

const char* ssm_last_plan(void) { return g_last_plan.c_str(); }

int ssm_version(void) { return kVersion; }

}  // extern "C"
