// ssm_host_api.cu -- the scan with host buffers (ssm_scan_fwd_host).
//
// The batch is cut into pieces (a batch row, or a range of its channels when there
// are few rows), and the pieces stream through a ring of three device staging
// slots: while piece p is scanned on the compute stream, piece p + 1's inputs
// arrive on the copy-in stream and piece p - 1's output leaves on the copy-out
// stream.  PCIe carries both directions at once, so a call costs about its
// host-to-device bytes over the link plus one piece's scan and copy-out.  Every
// copy is one cudaMemcpyAsync of a contiguous slice: u, delta, z, y rows of a piece
// are consecutive (b * dim + d), and B, C are the piece's batch row.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "ssm.h"
#include "ssm_host.cuh"

namespace {

using namespace ssm_host;

constexpr int kSlots = 3;
constexpr int kTargetPieces = 8;

struct HostPlan {
  int64_t rows_per_piece = 1;   // batch rows per piece (>= 1)
  int64_t chans_per_piece = 0;  // channels per piece within a row (== dim when whole rows)
  int64_t pieces = 0;
  size_t scan_ws = 0;           // scan workspace of one piece
  size_t off_params = 0, off_slots = 0, slot_bytes = 0, off_log = 0, total = 0;
  size_t o_u = 0, o_d = 0, o_z = 0, o_y = 0, o_B = 0, o_C = 0, o_h0 = 0, o_hl = 0;
};

// Pieces: whole batch rows when there are at least kTargetPieces rows; otherwise
// each row is cut into ranges of channels (multiples of 128) so that about
// kTargetPieces pieces stream.
HostPlan host_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ssm_dtype io,
                   bool has_z, bool has_h0, bool has_hl, ssm_algo algo) {
  HostPlan h;
  const size_t es = (io == SSM_DTYPE_BF16) ? 2 : 4;
  if (batch >= kTargetPieces) {
    h.rows_per_piece = (batch + kTargetPieces - 1) / kTargetPieces;
    h.chans_per_piece = dim;
  } else {
    const int64_t per_row = (kTargetPieces + batch - 1) / batch;
    int64_t c = (dim + per_row - 1) / per_row;
    c = (c + 127) / 128 * 128;
    h.rows_per_piece = 1;
    h.chans_per_piece = c < dim ? c : dim;
  }
  const int64_t row_groups = (batch + h.rows_per_piece - 1) / h.rows_per_piece;
  const int64_t chan_groups = (dim + h.chans_per_piece - 1) / h.chans_per_piece;
  h.pieces = row_groups * chan_groups;
  const int64_t pr = h.rows_per_piece, pc = h.chans_per_piece;
  h.scan_ws = round_up(ssm_scan_fwd_algo_workspace_size(pr, pc, dstate, seqlen, algo), 256);
  h.off_params = h.scan_ws;
  const size_t params = round_up(static_cast<size_t>(dim) * dstate * 4, 256) +
                        2 * round_up(static_cast<size_t>(dim) * 4, 256);
  h.off_slots = h.off_params + params;
  const size_t chan_bytes = round_up(static_cast<size_t>(pr * pc) * seqlen * es, 256);
  const size_t bc_bytes = round_up(static_cast<size_t>(pr) * dstate * seqlen * es, 256);
  const size_t st_bytes = round_up(static_cast<size_t>(pr * pc) * dstate * 4, 256);
  size_t o = 0;
  h.o_u = o; o += chan_bytes;
  h.o_d = o; o += chan_bytes;
  h.o_z = o; o += has_z ? chan_bytes : 0;
  h.o_y = o; o += chan_bytes;
  h.o_B = o; o += bc_bytes;
  h.o_C = o; o += bc_bytes;
  h.o_h0 = o; o += has_h0 ? st_bytes : 0;
  h.o_hl = o; o += has_hl ? st_bytes : 0;
  h.slot_bytes = o;
  h.off_log = h.off_slots + kSlots * h.slot_bytes;  // each piece's status words
  h.total = h.off_log + round_up(static_cast<size_t>(h.pieces) * sizeof(ssm::DeviceStatus), 256);
  return h;
}

struct Streams {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
  cudaEvent_t params_done = nullptr;
  bool ok = false;
  Streams() {
    ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&comp, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&params_done, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s)
      ok = cudaEventCreateWithFlags(&in_done[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&comp_done[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&out_done[s], cudaEventDisableTiming) == cudaSuccess;
  }
  // On every return path: no copy of this call may still be writing the caller's
  // host buffers (or reading them) once the call has returned.
  ~Streams() {
    if (in) cudaStreamSynchronize(in);
    if (comp) cudaStreamSynchronize(comp);
    if (out) cudaStreamSynchronize(out);
    for (int s = 0; s < kSlots; ++s) {
      if (in_done[s]) cudaEventDestroy(in_done[s]);
      if (comp_done[s]) cudaEventDestroy(comp_done[s]);
      if (out_done[s]) cudaEventDestroy(out_done[s]);
    }
    if (params_done) cudaEventDestroy(params_done);
    if (in) cudaStreamDestroy(in);
    if (comp) cudaStreamDestroy(comp);
    if (out) cudaStreamDestroy(out);
  }
};

}  // namespace

extern "C" {

size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                        int64_t seqlen, ssm_dtype io, int has_z, int has_h0,
                                        int has_h_last, ssm_algo algo) {
  if (batch < 1 || dim < 1 || dstate < 1 || seqlen < 1) return kStatusBytes;
  return host_plan(batch, dim, dstate, seqlen, io, has_z != 0, has_h0 != 0, has_h_last != 0,
                   algo)
      .total;
}

ssm_status ssm_scan_fwd_host(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             ssm_dtype io, const void* u, const void* delta,
                             const float* delta_bias, int delta_softplus, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* h0, float* h_last, void* y, void* workspace,
                             size_t workspace_bytes, ssm_discretization disc, ssm_algo algo) {
  ssm_status st = validate_common(batch, dim, dstate, io);
  if (st != SSM_OK) return st;
  if (seqlen < 1 || seqlen > INT32_MAX - 4096) return SSM_ERR_INVALID_ARG;
  if (batch > (int64_t(1) << 62) / dim / seqlen) return SSM_ERR_INVALID_ARG;
  if (!u || !delta || !A || !B || !C || !y || !workspace) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SSM_ERR_INVALID_ARG;
  const HostPlan h = host_plan(batch, dim, dstate, seqlen, io, z != nullptr, h0 != nullptr,
                               h_last != nullptr, algo);
  if (workspace_bytes < h.total) return SSM_ERR_INVALID_ARG;
  const size_t es = (io == SSM_DTYPE_BF16) ? 2 : 4;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  Streams s;
  if (!s.ok) return cuda_fail(cudaGetLastError(), "scan_fwd_host streams");

  // parameters, once: A [dim][N], D [dim], bias [dim]
  float* dA = reinterpret_cast<float*>(ws + h.off_params);
  float* dD = reinterpret_cast<float*>(ws + h.off_params +
                                       round_up(static_cast<size_t>(dim) * dstate * 4, 256));
  float* dbias = dD + round_up(static_cast<size_t>(dim) * 4, 256) / 4;
  cudaError_t e = cudaMemcpyAsync(dA, A, static_cast<size_t>(dim) * dstate * 4,
                                  cudaMemcpyHostToDevice, s.in);
  if (e == cudaSuccess && D)
    e = cudaMemcpyAsync(dD, D, static_cast<size_t>(dim) * 4, cudaMemcpyHostToDevice, s.in);
  if (e == cudaSuccess && delta_bias)
    e = cudaMemcpyAsync(dbias, delta_bias, static_cast<size_t>(dim) * 4, cudaMemcpyHostToDevice,
                        s.in);
  if (e == cudaSuccess) e = cudaEventRecord(s.params_done, s.in);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s.comp, s.params_done, 0);
  if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host parameters");

  const int64_t chan_groups = (dim + h.chans_per_piece - 1) / h.chans_per_piece;
  const unsigned char* hu = static_cast<const unsigned char*>(u);
  const unsigned char* hd = static_cast<const unsigned char*>(delta);
  const unsigned char* hz = static_cast<const unsigned char*>(z);
  const unsigned char* hB = static_cast<const unsigned char*>(B);
  const unsigned char* hC = static_cast<const unsigned char*>(C);
  unsigned char* hy = static_cast<unsigned char*>(y);
  for (int64_t p = 0; p < h.pieces; ++p) {
    const int slot = static_cast<int>(p % kSlots);
    unsigned char* sl = ws + h.off_slots + slot * h.slot_bytes;
    const int64_t b0 = (p / chan_groups) * h.rows_per_piece;
    const int64_t d0 = (p % chan_groups) * h.chans_per_piece;
    const int64_t nb = (batch - b0 < h.rows_per_piece) ? batch - b0 : h.rows_per_piece;
    const int64_t nd = (dim - d0 < h.chans_per_piece) ? dim - d0 : h.chans_per_piece;
    // rows of the piece: b0 .. b0+nb-1 with channels d0 .. d0+nd-1; contiguous in
    // [batch][dim][L] when the piece is whole rows (nd == dim) or a single row
    const int64_t row0 = b0 * dim + d0;
    const size_t chan_bytes = static_cast<size_t>(nb * nd) * seqlen * es;
    const size_t bc_bytes = static_cast<size_t>(nb) * dstate * seqlen * es;
    const size_t st_bytes = static_cast<size_t>(nb * nd) * dstate * 4;
    const size_t chan_off = static_cast<size_t>(row0) * seqlen * es;
    const size_t bc_off = static_cast<size_t>(b0) * dstate * seqlen * es;
    const size_t st_off = static_cast<size_t>(row0) * dstate * 4;

    // copy in, once the slot's previous piece has been copied out
    if (p >= kSlots) e = cudaStreamWaitEvent(s.in, s.out_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sl + h.o_u, hu + chan_off, chan_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sl + h.o_d, hd + chan_off, chan_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess && z)
      e = cudaMemcpyAsync(sl + h.o_z, hz + chan_off, chan_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sl + h.o_B, hB + bc_off, bc_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sl + h.o_C, hC + bc_off, bc_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess && h0)
      e = cudaMemcpyAsync(sl + h.o_h0, reinterpret_cast<const unsigned char*>(h0) + st_off,
                          st_bytes, cudaMemcpyHostToDevice, s.in);
    if (e == cudaSuccess) e = cudaEventRecord(s.in_done[slot], s.in);
    if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host copy in");

    // scan the piece
    e = cudaStreamWaitEvent(s.comp, s.in_done[slot], 0);
    if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host wait");
    st = ssm_scan_fwd_ex(nb, nd, dstate, seqlen, io, sl + h.o_u, sl + h.o_d,
                         delta_bias ? dbias + d0 : nullptr, delta_softplus, dA + d0 * dstate,
                         sl + h.o_B, sl + h.o_C, D ? dD + d0 : nullptr, z ? sl + h.o_z : nullptr,
                         h0 ? reinterpret_cast<const float*>(sl + h.o_h0) : nullptr,
                         h_last ? reinterpret_cast<float*>(sl + h.o_hl) : nullptr, sl + h.o_y,
                         ws, h.scan_ws, disc, algo, reinterpret_cast<ssm_stream_t>(s.comp));
    if (st != SSM_OK) return st;
    // keep the piece's status words (the next scan clears them)
    e = cudaMemcpyAsync(ws + h.off_log + p * sizeof(ssm::DeviceStatus), ws,
                        sizeof(ssm::DeviceStatus), cudaMemcpyDeviceToDevice, s.comp);
    if (e == cudaSuccess) e = cudaEventRecord(s.comp_done[slot], s.comp);

    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s.out, s.comp_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(hy + chan_off, sl + h.o_y, chan_bytes, cudaMemcpyDeviceToHost, s.out);
    if (e == cudaSuccess && h_last)
      e = cudaMemcpyAsync(reinterpret_cast<unsigned char*>(h_last) + st_off, sl + h.o_hl,
                          st_bytes, cudaMemcpyDeviceToHost, s.out);
    if (e == cudaSuccess) e = cudaEventRecord(s.out_done[slot], s.out);
    if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host copy out");
  }
  e = cudaStreamSynchronize(s.out);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s.comp);
  if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host synchronize");
  // device-side wait timeouts of any piece's scan
  for (int64_t p = 0; p < h.pieces; ++p) {
    ssm::DeviceStatus ds;
    e = cudaMemcpy(&ds, ws + h.off_log + p * sizeof(ssm::DeviceStatus), sizeof(ds),
                   cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_host status");
    if (ds.flags & ssm::kStatusTimeout) return SSM_ERR_DEVICE_TIMEOUT;
  }
  return SSM_OK;
}

}  // extern "C"
