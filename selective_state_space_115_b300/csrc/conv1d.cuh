// conv1d.cuh -- causal depthwise convolution over time (+ silu), the step before
// the scan in the MambaBlock of Mamba_Model_Report.md (section 3: conv1d with
// groups = channels, padding W - 1, the first L outputs, then silu), and its
// single-token form for decode (section 6: the cached W - 1 inputs plus the new
// one; the cache drops its oldest input).
//
//   out[b,d,l] = act(bias[d] + sum_{k<W} w[d,k] x[b,d,l-(W-1)+k])
//
// with x before position 0 taken from the carried-in window (or zero).  The pass
// reads x once and writes out once (memory-bound): a thread owns one 16-byte
// vector of positions of one row (8 bf16 / 4 fp32), takes the W - 1 inputs before
// it with scalar loads that hit L1 (its neighbour loaded them), and writes its
// outputs as one 16-byte vector.  Grid: x over runs of a row, y over rows.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

constexpr int kConvMaxWidth = 8;

struct ConvParams {
  int64_t row0;            // first row (b * dim + d) of this launch
  int64_t rows;            // rows in all
  int dim, seqlen, width;
  int silu;
  const void* x;           // [rows, seqlen]
  const float* w;          // [dim, width]
  const float* bias;       // [dim] or null
  const void* state_in;    // [rows, width - 1] or null: inputs before position 0
  void* out;               // [rows, seqlen] (decode: [rows])
  void* state_out;         // [rows, width - 1] or null: the last width - 1 inputs
  void* state;             // decode: [rows, width - 1], updated in place
  // aligned full-sequence kernel: vectors of this launch (< 2^31), the divisors
  // vectors-per-row and dim, and row0 % dim
  uint32_t nvec;
  FastDivU32 div_vpr, div_dim;
  uint32_t row0_mod;
};

// a 16-byte vector of io values to / from fp32
template <typename IO>
__device__ __forceinline__ void unpack16(const uint4 v, float* out) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  if constexpr (sizeof(IO) == 2) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = bf16lo(w4[k]);
      out[2 * k + 1] = bf16hi(w4[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = __uint_as_float(w4[k]);
  }
}
template <typename IO>
__device__ __forceinline__ uint4 pack16(const float* o) {
  if constexpr (sizeof(IO) == 2) {
    return make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                      pack_bf16x2(o[6], o[7]));
  } else {
    return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                      __float_as_uint(o[3]));
  }
}

template <typename IO>
__device__ __forceinline__ float conv_act(float v, int silu) {
  if (!silu) return v;
  return (sizeof(IO) == 2) ? silu_fast(v) : silu_accurate(v);
}

template <typename IO, bool VEC>
__global__ void __launch_bounds__(128) conv1d_fwd_kernel(const ConvParams p) {
  constexpr int TB = 16 / static_cast<int>(sizeof(IO));  // positions per thread
  const int64_t row = p.row0 + blockIdx.y;
  const int l0 = (blockIdx.x * 128 + threadIdx.x) * TB;
  if (l0 >= p.seqlen) return;
  const int W = p.width;
  const int d = static_cast<int>(row % p.dim);
  const IO* xr = static_cast<const IO*>(p.x) + row * p.seqlen;
  const IO* sr = p.state_in ? static_cast<const IO*>(p.state_in) + row * (W - 1) : nullptr;

  // window: positions l0 - (kConvMaxWidth - 1) .. l0 + TB - 1 (only the last W - 1 + TB used)
  float win[kConvMaxWidth - 1 + TB];
#pragma unroll
  for (int k = 0; k < kConvMaxWidth - 1; ++k) {
    const int pos = l0 - (kConvMaxWidth - 1) + k;
    float v = 0.0f;
    if (k >= kConvMaxWidth - W) {  // the W - 1 inputs a width-W filter reaches back to
      if (pos >= 0)
        v = Io<IO>::ldg(xr + pos);
      else if (sr && pos >= -(W - 1))
        v = Io<IO>::ldg(sr + (W - 1) + pos);
    }
    win[k] = v;
  }
  const bool full = l0 + TB <= p.seqlen;
  if (VEC && full) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + l0));
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    if constexpr (sizeof(IO) == 2) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        win[kConvMaxWidth - 1 + 2 * k] = bf16lo(w4[k]);
        win[kConvMaxWidth - 1 + 2 * k + 1] = bf16hi(w4[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) win[kConvMaxWidth - 1 + k] = __uint_as_float(w4[k]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < TB; ++j)
      win[kConvMaxWidth - 1 + j] = (l0 + j < p.seqlen) ? Io<IO>::ldg(xr + l0 + j) : 0.0f;
  }

  // taps aligned to the window's end: tap kk (of kConvMaxWidth) multiplies the input
  // kConvMaxWidth - 1 - kk positions back, so a width-W filter fills the last W
  float wk[kConvMaxWidth];
#pragma unroll
  for (int kk = 0; kk < kConvMaxWidth; ++kk) {
    const int k = kk - (kConvMaxWidth - W);
    wk[kk] = (k >= 0) ? __ldg(p.w + static_cast<int64_t>(d) * W + k) : 0.0f;
  }
  const float bias = p.bias ? __ldg(p.bias + d) : 0.0f;

  float o[TB];
#pragma unroll
  for (int j = 0; j < TB; ++j) {
    float acc = bias;
#pragma unroll
    for (int kk = 0; kk < kConvMaxWidth; ++kk) acc = fmaf(wk[kk], win[j + kk], acc);
    o[j] = conv_act<IO>(acc, p.silu);
  }
  IO* orow = static_cast<IO*>(p.out) + row * p.seqlen;
  if (VEC && full) {
    uint4 v;
    if constexpr (sizeof(IO) == 2) {
      v = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                     pack_bf16x2(o[6], o[7]));
    } else {
      v = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                     __float_as_uint(o[3]));
    }
    *reinterpret_cast<uint4*>(orow + l0) = v;
  } else {
#pragma unroll
    for (int j = 0; j < TB; ++j)
      if (l0 + j < p.seqlen) Io<IO>::store(orow + l0 + j, o[j]);
  }
  // the run holding position L - 1 writes the last W - 1 inputs (they all lie in
  // its window: positions L - (W-1) .. L - 1 >= l0 - (W-1))
  if (p.state_out && l0 + TB >= p.seqlen) {
    IO* so = static_cast<IO*>(p.state_out) + row * (W - 1);
#pragma unroll
    for (int k = 0; k < kConvMaxWidth - 1; ++k) {
      if (k < W - 1) {
        const int pos = p.seqlen - (W - 1) + k;           // absolute position
        const int idx = (kConvMaxWidth - 1) + (pos - l0);  // window index
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < kConvMaxWidth - 1 + TB; ++t)
          if (t == idx) v = win[t];
        Io<IO>::store(so + k, v);
      }
    }
  }
}

// Aligned rows (seqlen * esize a multiple of 16, 16-byte aligned x and out): the
// rows are cut into 16-byte vectors of TB positions, numbered row-major, and a
// CTA of 128 threads takes the U * 128 consecutive vectors from base, thread t
// vector base + u*128 + t.  All U loads are issued before any arithmetic (U
// vectors in flight per thread) and parked in shared memory with the NPREV
// vectors just before the CTA's, so the W - 1 inputs before each vector come from
// shared memory; only vectors at the start of a row read the carried state (or
// zero).  The filter width is a template argument: each output costs exactly W
// multiply-adds.
template <typename IO, int W>
__global__ void __launch_bounds__(128) conv1d_fwd_vec_kernel(const ConvParams p) {
  constexpr int TB = 16 / static_cast<int>(sizeof(IO));  // positions per vector
  constexpr int NPREV = (W - 1 + TB - 1) / TB;            // previous vectors a window needs
  constexpr int U = 4;
  constexpr int WIN = (NPREV + 1) * TB;
  __shared__ __align__(16) uint4 sv[NPREV + 128 * U];
  // launched with programmatic stream serialisation: wait for the previous kernel
  // on the stream (and its writes) before reading x, then let the next one launch
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tid = threadIdx.x;
  const uint32_t vpr = p.div_vpr.d;  // vectors per row
  const uint32_t cta0 = blockIdx.x * (128u * U);
  const IO* x = static_cast<const IO*>(p.x) + p.row0 * p.seqlen;
  // vectors of the launch are contiguous: vector e starts at element e * TB

  uint4 cur[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t e = cta0 + u * 128 + tid;
    cur[u] = (e < p.nvec) ? __ldg(reinterpret_cast<const uint4*>(x) + e)
                          : make_uint4(0u, 0u, 0u, 0u);
  }
  if (NPREV > 0 && tid < NPREV) {
    const int64_t e = static_cast<int64_t>(cta0) - NPREV + tid;
    sv[tid] = (e >= 0 && e < p.nvec) ? __ldg(reinterpret_cast<const uint4*>(x) + e)
                                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) sv[NPREV + u * 128 + tid] = cur[u];
  __syncthreads();

#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t e = cta0 + u * 128 + tid;
    if (e >= p.nvec) break;
    const uint32_t rl = p.div_vpr.div(e);  // row within the launch
    const uint32_t v = e - rl * vpr;       // vector within the row
    const int64_t row = p.row0 + rl;
    const int l0 = static_cast<int>(v) * TB;
    float win[WIN];
#pragma unroll
    for (int k = NPREV; k >= 1; --k) {
      float* dst = win + (NPREV - k) * TB;
      if (v >= static_cast<uint32_t>(k)) {
        unpack16<IO>(sv[NPREV + u * 128 + tid - k], dst);
      } else {
        // before position 0: the carried-in inputs, or zero
        const IO* sr = p.state_in ? static_cast<const IO*>(p.state_in) + row * (W - 1) : nullptr;
#pragma unroll
        for (int j = 0; j < TB; ++j) {
          const int pos = l0 - k * TB + j;
          dst[j] = (sr && pos >= -(W - 1)) ? Io<IO>::ldg(sr + (W - 1) + pos) : 0.0f;
        }
      }
    }
    unpack16<IO>(cur[u], win + NPREV * TB);

    const uint32_t rd = p.row0_mod + rl;
    const uint32_t d = rd - p.div_dim.div(rd) * p.div_dim.d;  // row % dim
    float wk[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wk[k] = __ldg(p.w + d * W + k);
    const float bias = p.bias ? __ldg(p.bias + d) : 0.0f;
    float o[TB];
    if constexpr (sizeof(IO) == 2) {
      // outputs in pairs, packed f32x2: the same multiply-adds in the same order as
      // the scalar form (bit-identical sums) in half the instructions; silu(v) =
      // h + h tanh(h) with h = v / 2 (the hardware tanh, as silu_fast)
      f2 acc2[TB / 2];
#pragma unroll
      for (int q = 0; q < TB / 2; ++q) acc2[q] = mk2(bias, bias);
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const f2 w2 = mk2(wk[k], wk[k]);
#pragma unroll
        for (int q = 0; q < TB / 2; ++q) {
          const int i0 = NPREV * TB + 2 * q - (W - 1) + k;
          acc2[q] = fma2(w2, mk2(win[i0], win[i0 + 1]), acc2[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < TB / 2; ++q) {
        f2 v = acc2[q];
        if (p.silu) {
          const f2 h = mul2(v, mk2(0.5f, 0.5f));
          v = fma2(h, mk2(tanh_hw(h.x), tanh_hw(h.y)), h);
        }
        o[2 * q] = v.x;
        o[2 * q + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < TB; ++j) {
        float acc = bias;
#pragma unroll
        for (int k = 0; k < W; ++k) acc = fmaf(wk[k], win[NPREV * TB + j - (W - 1) + k], acc);
        o[j] = conv_act<IO>(acc, p.silu);
      }
    }
    reinterpret_cast<uint4*>(static_cast<IO*>(p.out) + p.row0 * p.seqlen)[e] = pack16<IO>(o);
    if (p.state_out && v == vpr - 1) {
      IO* so = static_cast<IO*>(p.state_out) + row * (W - 1);
#pragma unroll
      for (int k = 0; k < W - 1; ++k) Io<IO>::store(so + k, win[NPREV * TB + TB - (W - 1) + k]);
    }
  }
}

// One decode position per (batch, dim) channel; the cache p.state [rows, W-1] is
// updated in place.
template <typename IO>
__global__ void __launch_bounds__(256) conv1d_update_kernel(const ConvParams p) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (row >= p.rows) return;
  const int W = p.width;
  const int d = static_cast<int>(row % p.dim);
  IO* s = static_cast<IO*>(p.state) + row * (W - 1);
  float win[kConvMaxWidth - 1];
#pragma unroll
  for (int k = 0; k < kConvMaxWidth - 1; ++k) win[k] = (k < W - 1) ? Io<IO>::load(s + k) : 0.0f;
  const IO xraw = static_cast<const IO*>(p.x)[row];
  const float xv = Io<IO>::load(&xraw);
  float acc = p.bias ? __ldg(p.bias + d) : 0.0f;
#pragma unroll
  for (int k = 0; k < kConvMaxWidth - 1; ++k)
    if (k < W - 1) acc = fmaf(__ldg(p.w + static_cast<int64_t>(d) * W + k), win[k], acc);
  acc = fmaf(__ldg(p.w + static_cast<int64_t>(d) * W + W - 1), xv, acc);
  Io<IO>::store(static_cast<IO*>(p.out) + row, conv_act<IO>(acc, p.silu));
  // drop the oldest input, append x as given (the cache holds the raw inputs)
#pragma unroll
  for (int k = 0; k + 1 < kConvMaxWidth - 1; ++k)
    if (k + 1 < W - 1) s[k] = s[k + 1];
  if (W > 1) s[W - 2] = xraw;
}

}  // namespace ssm
