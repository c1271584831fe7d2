/*
 * ssm.h -- C ABI of libssm: the Mamba selective-scan forward and the
 * single-token recurrent state update, as CUDA kernels for B300 (sm_103a).
 *
 * The method (citations are to the pages this library follows):
 *
 *   dt_l   = softplus(delta[b,d,l] + delta_bias[d])            (or no softplus)
 *   Abar   = exp(dt_l * A[d,n])
 *   Bbar   = (dt_l A)^-1 (exp(dt_l A) - 1) dt_l B[b,n,l]  = (Abar - 1) / A[d,n] * B[b,n,l]
 *            (= dt_l * B[b,n,l] when A[d,n] == 0, the A -> 0 limit)
 *   h_l[n] = Abar * h_{l-1}[n] + Bbar * u[b,d,l]                h_{-1} = h0 (or 0)
 *   y_l    = sum_n C[b,n,l] * h_l[n] + D[d] * u[b,d,l]
 *   y_l   *= silu(z[b,d,l])                                     (when z is given)
 *
 *  - zero-order-hold discretisation and the recurrence h_k = Abar h_{k-1} + Bbar x_k:
 *    velog review of "Mamba: Linear-Time Sequence Modeling with Selective State
 *    Spaces", section 2 "Discretization"; the ZOH integral and the need for an
 *    invertible A: "mamba 学习" (fakeeyes2wo), section "MAMBA".
 *  - input-dependent dt, B, C and A fixed per channel: velog review, sections
 *    3.2 and 3.5; "Mamba学习记录" (lengnian), section "怎么增加选择性".
 *  - D skip and silu(z) gate: Mamba_Model_Report.md, sections 3 and 4.2.
 *  - single-token step: Mamba_Model_Report.md, section 6 (ssm_step).
 *  - fusion rule (load the 3-D inputs once, keep the state on chip, write only
 *    the 3-D output; never materialise the (B, L, D, N) tensor): velog review,
 *    section 3.3 "Kernel Fusion".
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers, owned by the caller.  The library
 *    allocates no device memory and keeps no per-call state -- except
 *    ssm_scan_fwd_noalloc, whose statically reserved scratch keeps the last call's
 *    contents (see its comment).
 *  - Tensors are contiguous, row-major, last index fastest:
 *      u, delta, z, y : [batch, dim, seqlen]      (scan)  /  [batch, dim]  (update)
 *      B, C           : [batch, dstate, seqlen]   (scan)  /  [batch, dstate] (update)
 *      A              : [dim, dstate]     float32
 *      D, delta_bias  : [dim]             float32
 *      h0, h_last, h  : [batch, dim, dstate] float32
 *  - u, delta, z, B, C and y have the io dtype (float32 or bfloat16); A, D,
 *    delta_bias and every state tensor are float32.  Arithmetic is float32.
 *    bfloat16 outputs are rounded to nearest even.
 *  - dstate must be 4, 8 or 16 (SSM_ERR_UNSUPPORTED otherwise).  batch, dim and
 *    seqlen may be any value >= 1; there is no alignment requirement beyond the
 *    element size (aligned, L-multiple shapes take the TMA path).
 *  - Arguments are validated on the host before anything is enqueued; a call
 *    that returns an error has launched nothing.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and the call returns without synchronising.  A launch failure returns
 *    SSM_ERR_CUDA (ssm_last_cuda_error() gives the CUDA message).
 *  - Outputs must not alias inputs, except that ssm_state_update updates h in place.
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same ABI as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* ssm_stream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,    /* bad size, NULL required pointer, misaligned pointer */
    SSM_ERR_UNSUPPORTED = 2,    /* valid but not built: dstate not in {4, 8, 16}, unknown dtype/algo */
    SSM_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
    SSM_ERR_DEVICE_TIMEOUT = 4  /* a bounded device-side wait gave up (see ssm_read_device_status) */
} ssm_status;

typedef enum { SSM_DTYPE_F32 = 0, SSM_DTYPE_BF16 = 1 } ssm_dtype;

/* Input term of the discretisation (Abar = exp(dt A) in both):
 *   ZOH   Bbar = (exp(dt A) - 1) / A * B  (dt B where A == 0): the zero-order hold of
 *         the velog review, section 2 "Discretization" -- the default;
 *   EULER Bbar = dt * B: the form Mamba_Model_Report.md, section 4.2 (selective_scan:
 *         deltaB = delta * B) computes. */
typedef enum { SSM_DISC_ZOH = 0, SSM_DISC_EULER = 1 } ssm_discretization;

/* Kernel family of the scan.  AUTO picks by the number of independent
 * (batch, dim) channels: many channels -> CHANNEL, few -> CHUNK. */
typedef enum {
    SSM_ALGO_AUTO = 0,
    SSM_ALGO_CHANNEL = 1,     /* lanes over channels; 1, 2 or 4 adjacent lanes run a
                                 channel's whole sequence, each with a slice of its
                                 states in registers; L streamed through shared memory
                                 in TMA chunks.  The lanes-per-channel split is chosen
                                 from the sizes (finer split = more, shorter warps) */
    SSM_ALGO_CHUNK = 2,       /* lanes over positions; warp-shuffle associative scan of
                                 (Abar, Bbar u) pairs inside each chunk, state carried
                                 across chunks */
    SSM_ALGO_CHANNEL_L1 = 3,  /* CHANNEL with a fixed split: 1 lane per channel */
    SSM_ALGO_CHANNEL_L2 = 4,  /* 2 lanes per channel (dstate 8 or 16) */
    SSM_ALGO_CHANNEL_L4 = 5,  /* 4 lanes per channel (dstate 16) */
    SSM_ALGO_SEGMENTED = 6    /* long sequences over few channels: the sequence is split
                                 into segments run by separate CTAs (one lane per
                                 channel) in two passes -- each segment's end state from
                                 a zero state, then every segment again from the state
                                 rebuilt from the earlier segments.  Needs the workspace
                                 that ssm_scan_fwd_workspace_size() reports; sequences
                                 too short to split run as CHANNEL_L1 */,
    SSM_ALGO_CHANNEL_MIXED = 7 /* dstate 16: every SM runs the same number k of
                                 one-lane-per-channel CTAs of 128 channels, and the
                                 tiles left over run as 32-channel CTAs with four lanes
                                 per channel (each CTA takes its role when it starts;
                                 the splits give identical bits).  CHANNEL picks it when
                                 its cost model favours it; other dstate run CHANNEL */
} ssm_algo;

/*
 * Size in bytes of the device workspace ssm_scan_fwd needs for these sizes on
 * the current device: 256 bytes of device status words, plus, when the sequence
 * is long and the channels few (the segmented plan), each segment's fp32 end
 * state and step-size sum.  A smaller workspace (at least 256 bytes) is accepted
 * by SSM_ALGO_AUTO, which then runs a plan that fits it.
 */
SSM_API size_t ssm_scan_fwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen);

/* Workspace bytes ssm_scan_fwd_algo needs with this kernel family (AUTO: the same
 * as ssm_scan_fwd_workspace_size; SEGMENTED: room for at least two segments;
 * every other family: the 256 bytes of status words). */
SSM_API size_t ssm_scan_fwd_algo_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                                int64_t seqlen, ssm_algo algo);

/*
 * Selective-scan forward over a whole sequence (the pages' selective scan with
 * ZOH discretisation, fused: softplus, discretisation, recurrence,
 * C-contraction, D skip and gate in one kernel; u, delta, z, B, C read once,
 * y written once).
 *
 *  io             dtype of u, delta, z, B, C, y
 *  u, delta, y    [batch, dim, seqlen], required
 *  delta_bias     [dim] float32 or NULL (0)
 *  delta_softplus nonzero: dt = softplus(delta + bias); zero: dt = delta + bias
 *  A              [dim, dstate] float32, required (A == 0 entries use the dt limit)
 *  B, C           [batch, dstate, seqlen], required
 *  D              [dim] float32 or NULL (no skip)
 *  z              [batch, dim, seqlen] or NULL (no gate)
 *  h0             [batch, dim, dstate] float32 or NULL (zero initial state)
 *  h_last         [batch, dim, dstate] float32 or NULL (final state not written)
 *  workspace      device buffer of at least ssm_scan_fwd_workspace_size() bytes,
 *                 16-byte aligned, required.  Its status words are cleared on
 *                 `stream` before the kernel runs; a device-side wait that hits
 *                 its iteration limit records SSM_ERR_DEVICE_TIMEOUT there (the
 *                 outputs are then incomplete).  Calls that share a workspace
 *                 must not overlap on the GPU.
 * Returns SSM_OK once the work is enqueued.
 */
SSM_API ssm_status ssm_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ssm_dtype io,
                        const void* u, const void* delta, const float* delta_bias,
                        int delta_softplus, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* h0, float* h_last, void* y,
                        void* workspace, size_t workspace_bytes, ssm_stream_t stream);

/* ssm_scan_fwd with an explicit kernel family (SSM_ALGO_AUTO behaves exactly
 * like ssm_scan_fwd).  The CHANNEL variants fall back to CHUNK when the TMA
 * alignment rules do not hold (seqlen * element size not a multiple of 16, or a
 * tensor base not 16-byte aligned); a fixed lanes-per-channel split that would
 * leave a lane fewer than 4 states (L2 with dstate 4, L4 with dstate 4 or 8)
 * returns SSM_ERR_UNSUPPORTED. */
SSM_API ssm_status ssm_scan_fwd_algo(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             ssm_dtype io, const void* u, const void* delta,
                             const float* delta_bias, int delta_softplus, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* h0, float* h_last, void* y, void* workspace,
                             size_t workspace_bytes, ssm_algo algo, ssm_stream_t stream);

/* ssm_scan_fwd_algo with an explicit discretisation of the input term (ssm_scan_fwd
 * and ssm_scan_fwd_algo use SSM_DISC_ZOH).  Every kernel family supports both. */
SSM_API ssm_status ssm_scan_fwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                   ssm_dtype io, const void* u, const void* delta,
                                   const float* delta_bias, int delta_softplus, const float* A,
                                   const void* B, const void* C, const float* D, const void* z,
                                   const float* h0, float* h_last, void* y, void* workspace,
                                   size_t workspace_bytes, ssm_discretization disc,
                                   ssm_algo algo, ssm_stream_t stream);

/*
 * ssm_scan_fwd for callers that cannot allocate device memory, such as code
 * running under an allocator it does not own (a custom arena, a memory pool that
 * forbids new reservations) or inside a region where cudaMalloc is not allowed.
 * The pages have no counterpart to this entry point; it exists only for such
 * callers.  It allocates nothing: instead of a caller-provided workspace it uses
 * a scratch array of 4096 bytes reserved statically in the library, which every
 * GPU that loads the library keeps until the process exits.  The caller still
 * passes all inputs and outputs, exactly as for ssm_scan_fwd (kernel chosen as
 * by SSM_ALGO_AUTO).
 *  - The first call on a device (and the first after that device's context was
 *    reset or created again) looks up the scratch address (cudaGetSymbolAddress)
 *    with the caller's current device, which must be the device of the tensors
 *    and of `stream`; make that first call before any stream capture.
 *  - The kernel is chosen as by SSM_ALGO_AUTO among the plans whose scratch fits
 *    the reserved 4096 bytes: the channel kernels always fit; the segmented
 *    long-sequence plan is taken when its segment states fit (e.g. one channel of
 *    8192+ positions), and otherwise the lanes-over-positions kernel takes its
 *    place.  No size is rejected for want of scratch.
 *  - Every call shares the one array per device and it keeps the last call's
 *    contents; its status words are cleared on `stream` before each kernel.
 *    Calls that overlap on the GPU (different streams, no ordering) race on it.
 *  - Device-side wait timeouts are recorded in that shared array and are not
 *    reported back by this entry point.
 */
SSM_API ssm_status ssm_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                        ssm_dtype io, const void* u, const void* delta,
                                        const float* delta_bias, int delta_softplus,
                                        const float* A, const void* B, const void* C,
                                        const float* D, const void* z, const float* h0,
                                        float* h_last, void* y, ssm_stream_t stream);

/*
 * Single-token recurrent state update (decode): one step of the scan for every
 * (batch, dim) channel, h read and written in place (Mamba_Model_Report.md,
 * section 6, ssm_step, with the ZOH discretisation above).
 *
 *  h       [batch, dim, dstate] float32, in/out, required
 *  u, delta, y  [batch, dim], required;  z [batch, dim] or NULL
 *  B, C    [batch, dstate], required;  A [dim, dstate] float32, required
 *  delta_bias, D  [dim] float32 or NULL
 * No workspace: the kernel has no device-side waits.
 */
SSM_API ssm_status ssm_state_update(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io, float* h,
                            const void* u, const void* delta, const float* delta_bias,
                            int delta_softplus, const float* A, const void* B, const void* C,
                            const float* D, const void* z, void* y, ssm_stream_t stream);

/* ssm_state_update with an explicit discretisation of the input term. */
SSM_API ssm_status ssm_state_update_ex(int64_t batch, int64_t dim, int64_t dstate, ssm_dtype io,
                                       float* h, const void* u, const void* delta,
                                       const float* delta_bias, int delta_softplus,
                                       const float* A, const void* B, const void* C,
                                       const float* D, const void* z, void* y,
                                       ssm_discretization disc, ssm_stream_t stream);

/*
 * Gradient of ssm_scan_fwd (reverse mode), for training.
 *
 * Given dy = dLoss/dy [batch, dim, seqlen] (and optionally dh_last =
 * dLoss/dh_last [batch, dim, dstate]), returns the gradients of every input of
 * the scan: Mamba_Model_Report.md section 4.1 builds the recurrence's backward
 * from a reverse scan (pscan_rev) over the adjoint g_l = dLoss/dh_l, and
 * "Mamba学习记录" (lengnian), Part3, lists recomputation of intermediate results
 * among the hardware-aware algorithm's means: the states are recomputed from
 * checkpoints here, not stored by the forward pass.
 *
 *  forward inputs   exactly as passed to ssm_scan_fwd (u, delta, delta_bias,
 *                   delta_softplus, A, B, C, D, z, h0; same dtypes and layouts)
 *  dy               [batch, dim, seqlen] io dtype, required
 *  dh_last          [batch, dim, dstate] float32 or NULL (zero)
 *  du, ddelta       [batch, dim, seqlen] io dtype, required (overwritten)
 *  dA               [dim, dstate] float32, required
 *  dB, dC           [batch, dstate, seqlen] io dtype, required
 *  dD               [dim] float32; required iff D is given, else ignored
 *  dz               [batch, dim, seqlen] io dtype; required iff z is given
 *  ddelta_bias      [dim] float32 or NULL (not computed)
 *  dh0              [batch, dim, dstate] float32 or NULL (not computed)
 *  workspace        ssm_scan_bwd_workspace_size(...) bytes, 256-byte aligned;
 *                   its contents need not be preserved between calls
 *  disc             the discretisation the forward used
 *
 * Outputs must not overlap inputs or each other.  The reductions over channels
 * (dB, dC) and over batch rows and positions (dA, dD, ddelta_bias) are summed in
 * a fixed order: results are bit-reproducible for a given shape.  Arithmetic is
 * fp32; bf16 outputs are rounded to nearest even.  Validated on the host first
 * (nothing is enqueued when a check fails); enqueued on `stream`.
 *
 * The state checkpoints (every 8 positions, in the workspace) come from the
 * forward's own kernels in a checkpoint-only pass (no output, neither C nor z read)
 * when AUTO would run the forward on its channel kernel, mixed split or segmented
 * plan (with `segments` 0), else from a forward pass of the gradient kernel; the
 * gradient is then bit for bit the one ssm_scan_bwd_ckpt returns from the
 * checkpoints of a training forward that ran AUTO's plan.  That pass records its wait
 * timeouts in the workspace's first 16 bytes, which ssm_read_device_status reads.
 */
SSM_API size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                           int64_t seqlen);
/*
 * ssm_scan_bwd with an explicit split of the sequence into `segments` pieces (0:
 * the library's choice; the choice splits only when the (batch row, 32-channel)
 * CTAs cannot fill the GPU, e.g. long sequences over few channels).  A split adds
 * a first pass per segment (its end state from a zero state, its own adjoint from a
 * zero adjoint, its step-size sum); the second pass combines them into each
 * segment's entering state and end adjoint, as the segmented forward does.
 * Results agree with the unsplit gradient up to rounding.  Negative `segments`
 * is SSM_ERR_INVALID_ARG; more segments than 8-position blocks are capped.
 */
SSM_API size_t ssm_scan_bwd_ex_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                              int64_t seqlen, int segments);
SSM_API ssm_status ssm_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                ssm_dtype io, const void* u, const void* delta,
                                const float* delta_bias, int delta_softplus, const float* A,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* h0, const void* dy, const float* dh_last, void* du,
                                void* ddelta, float* dA, void* dB, void* dC, float* dD, void* dz,
                                float* ddelta_bias, float* dh0, void* workspace,
                                size_t workspace_bytes, ssm_discretization disc,
                                ssm_stream_t stream);
SSM_API ssm_status ssm_scan_bwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                   ssm_dtype io, const void* u, const void* delta,
                                   const float* delta_bias, int delta_softplus, const float* A,
                                   const void* B, const void* C, const float* D, const void* z,
                                   const float* h0, const void* dy, const float* dh_last,
                                   void* du, void* ddelta, float* dA, void* dB, void* dC,
                                   float* dD, void* dz, float* ddelta_bias, float* dh0,
                                   void* workspace, size_t workspace_bytes,
                                   ssm_discretization disc, int segments, ssm_stream_t stream);

/*
 * Training step: the forward writes the state checkpoints the gradient needs, so the
 * gradient runs no forward pass of its own.  The pages' recomputation (lengnian,
 * Part3: intermediate states recomputed in the backward pass instead of stored) keeps
 * one fp32 state per channel every 8 positions (4 bytes per state every 8 positions:
 * the (B, L, D, N) tensor is never stored).
 *
 * ssm_scan_ckpt_bytes: bytes of the checkpoints, ceil(seqlen / 8) * batch * dim *
 * dstate * 4 (0 for invalid sizes).
 *
 * ssm_scan_fwd_train: ssm_scan_fwd_ex (same arguments, same y and h_last, bit for
 * bit) that also writes ckpt[j][b * dim + d][n] = the state entering position 8 j
 * (j = 0 .. ceil(seqlen / 8) - 1; j = 0 holds h0, or 0), float32, device memory owned
 * by the caller, 16-byte aligned, ckpt_bytes >= ssm_scan_ckpt_bytes().
 * SSM_ERR_INVALID_ARG for a NULL, misaligned or short buffer.
 *
 * ssm_scan_bwd_ckpt: ssm_scan_bwd_ex from those checkpoints (`ckpt`, as the training
 * forward wrote them for the same inputs and h0; float32, 4-byte aligned); workspace
 * of ssm_scan_bwd_ckpt_workspace_size() bytes (no room for checkpoints of its own).
 * The gradient equals ssm_scan_bwd_ex's up to the rounding of the states the two
 * forwards compute.
 */
SSM_API size_t ssm_scan_ckpt_bytes(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen);
SSM_API ssm_status ssm_scan_fwd_train(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                      ssm_dtype io, const void* u, const void* delta,
                                      const float* delta_bias, int delta_softplus,
                                      const float* A, const void* B, const void* C,
                                      const float* D, const void* z, const float* h0,
                                      float* h_last, void* y, float* ckpt, size_t ckpt_bytes,
                                      void* workspace, size_t workspace_bytes,
                                      ssm_discretization disc, ssm_algo algo,
                                      ssm_stream_t stream);
SSM_API size_t ssm_scan_bwd_ckpt_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                                int64_t seqlen, int segments);
SSM_API ssm_status ssm_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                     ssm_dtype io, const void* u, const void* delta,
                                     const float* delta_bias, int delta_softplus, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     const float* h0, const float* ckpt, const void* dy,
                                     const float* dh_last, void* du, void* ddelta, float* dA,
                                     void* dB, void* dC, float* dD, void* dz,
                                     float* ddelta_bias, float* dh0, void* workspace,
                                     size_t workspace_bytes, ssm_discretization disc,
                                     int segments, ssm_stream_t stream);

/*
 * Causal depthwise convolution over time, the step before the scan in the
 * MambaBlock of Mamba_Model_Report.md (section 3: nn.Conv1d with groups = channels,
 * kernel_size = width, padding = width - 1, the first L outputs, then silu):
 *
 *   out[b,d,l] = act(bias[d] + sum_{k<width} weight[d,k] * x[b,d,l-(width-1)+k])
 *
 * with act = silu (apply_silu != 0) or the identity, and x before position 0 taken
 * from conv_state (the width - 1 inputs that precede the sequence) or zero.
 *
 *  io           dtype of x, out and the two states (float32 or bfloat16)
 *  x, out       [batch, dim, seqlen], required; must not overlap
 *  weight       [dim, width] float32, required;  bias [dim] float32 or NULL
 *  conv_state   [batch, dim, width - 1] or NULL (zero history)
 *  conv_state_out [batch, dim, width - 1] or NULL: receives the last width - 1
 *               inputs (the decode cache; section 6 of the report)
 *  width        1 .. 8 (SSM_ERR_UNSUPPORTED otherwise)
 * Arithmetic is fp32; bf16 outputs are rounded to nearest even.  Validated on the
 * host first; enqueued on `stream`; no workspace, no device-side waits.
 */
SSM_API ssm_status ssm_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                                  ssm_dtype io, const void* x, const float* weight,
                                  const float* bias, const void* conv_state, int apply_silu,
                                  void* out, void* conv_state_out, ssm_stream_t stream);

/*
 * One decode position of the convolution above (Mamba_Model_Report.md section 6,
 * step): the window is conv_state[b,d,:] (the last width - 1 inputs) followed by
 * x[b,d]; out[b,d] = act(bias[d] + sum_k weight[d,k] window[k]); conv_state drops
 * its oldest input and appends x (in place).
 *  conv_state [batch, dim, width - 1] io dtype, in/out;  x, out [batch, dim]
 */
SSM_API ssm_status ssm_conv1d_update(int64_t batch, int64_t dim, int64_t width, ssm_dtype io,
                                     void* conv_state, const void* x, const float* weight,
                                     const float* bias, int apply_silu, void* out,
                                     ssm_stream_t stream);

/*
 * Synchronises `stream`, then reads the status words of `workspace` (as filled
 * by the last ssm_scan_fwd, or ssm_scan_bwd's checkpoint pass, that used it).
 * Returns SSM_OK, SSM_ERR_DEVICE_TIMEOUT, or SSM_ERR_CUDA if the synchronisation or
 * the copy failed.
 */
SSM_API ssm_status ssm_read_device_status(const void* workspace, ssm_stream_t stream);

/*
 * The scan with HOST buffers: u, delta, z, B, C, y, A, D, delta_bias, h0, h_last
 * as in ssm_scan_fwd_ex but in host memory (page-locked memory lets the copies
 * overlap; pageable memory works, without overlap).  The batch is cut into pieces
 * (a batch row, or a range of a row's channels when there are few rows) that
 * stream through three device staging slots in `workspace`: each piece is copied
 * in while the previous one is scanned and the one before it copied out, on
 * streams of the call's own, so the call costs about its host-to-device bytes over
 * the link.  Blocks until y (and h_last) hold the results.  Returns
 * SSM_ERR_DEVICE_TIMEOUT if any piece's scan recorded a timeout.
 *  workspace  device memory, ssm_scan_fwd_host_workspace_size(...) bytes, 256-byte
 *             aligned; `has_z`, `has_h0`, `has_h_last` say whether those are given
 */
SSM_API size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                                int64_t seqlen, ssm_dtype io, int has_z,
                                                int has_h0, int has_h_last, ssm_algo algo);
SSM_API ssm_status ssm_scan_fwd_host(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                     ssm_dtype io, const void* u, const void* delta,
                                     const float* delta_bias, int delta_softplus,
                                     const float* A, const void* B, const void* C,
                                     const float* D, const void* z, const float* h0,
                                     float* h_last, void* y, void* workspace,
                                     size_t workspace_bytes, ssm_discretization disc,
                                     ssm_algo algo);

/*
 * Check of the device-side timeout path: one CTA waits, with the library's
 * bounded wait and a limit of `limit_ns` nanoseconds (1e3 .. 1e10), for an
 * mbarrier phase that only completes when `arrive` is nonzero.  Without the
 * arrival the wait gives up and the kernel records the timeout in the status words
 * at the start of `workspace` (>= 16 bytes, 16-byte aligned, zeroed by the caller
 * beforehand); ssm_read_device_status then returns SSM_ERR_DEVICE_TIMEOUT.  The
 * kernel always returns normally and the context stays usable.
 */
SSM_API ssm_status ssm_selftest_wait(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                     int arrive, ssm_stream_t stream);

/* Static description of a status code. */
SSM_API const char* ssm_status_string(ssm_status status);

/* Detail of the last CUDA error (or rejected no-alloc request) seen by a call on
 * this host thread ("" if none). */
SSM_API const char* ssm_last_cuda_error(void);

/* Which kernels the last successful scan-forward call on this host thread launched
 * (ssm_scan_fwd, _algo, _ex, _noalloc), with the split the library chose, e.g.
 * "scan_channel_mixed_kernel: 2 one-lane CTAs per SM + 96 four-lane CTAs" ("" before
 * the first call).  A diagnostic for benchmarks and profiles; the text is not a
 * stable interface.  The pages have no counterpart. */
SSM_API const char* ssm_last_plan(void);

/* Library version: major * 10000 + minor * 100 + patch. */
SSM_API int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
