// scan_chunk.cuh -- selective-scan forward, "chunk" kernel family.
//
// For inputs with few (batch, dim) channels (long sequences, small layers),
// one warp owns one channel and splits each chunk of 32*T positions over its
// lanes (T consecutive positions per lane).  The recurrence h_l = Abar_l h_{l-1}
// + Bbar_l u_l is associative in the pairs (Abar, Bbar u):
//     (P1, H1) then (P2, H2)  =  (P1 P2, P2 H1 + H2)
// (velog Mamba review, section 3.3 "Parallel Scan"), so per state n each lane
//   1. forms its T pairs and folds them into one (P, H) (zero initial state),
//   2. joins a 5-step warp-shuffle inclusive scan of (P, H) over the lanes,
//   3. takes its carry-in h = P_prev * h_chunk + H_prev from the exclusive
//      prefix and replays its T positions, accumulating y += C h,
// and the state after the last lane is carried (in shared memory) to the next chunk.
// The 4-D (position, state) tensor exists only as T pairs per lane per state.
//
// A CTA holds WARPS (8) channels of one batch row, which share B and C: each chunk's B
// and C tiles ([N][32*T] each) are staged once per CTA in shared memory (cp.async,
// one chunk ahead, when rows are 16-byte aligned; element loads otherwise), so the
// per-state loop reads them from shared memory instead of waiting on global loads.
// u, delta and z are plain coalesced global loads, so this kernel accepts every
// shape and alignment.
#pragma once

#include "scan_channel.cuh"
#include "ssm_device.cuh"

namespace ssm {

template <typename IO, int N_, bool GATE_, bool VEC_, bool EULER_ = false>
struct ChunkCfg {
  static constexpr int N = N_;
  static constexpr bool GATE = GATE_;
  static constexpr bool EULER = EULER_;     // input term dt * B instead of the ZOH form
  static constexpr bool VEC = VEC_;
  // 8 channels per CTA: the CTAs of a 3072-channel layer (the 130M-like one) then
  // fit the SMs in one wave (3 per SM by the 64 KB of B, C staging); at 4 channels
  // they took 1.73 waves (measured on B300: 148 -> 124 us)
  static constexpr int WARPS = 8;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int ESZ = Io<IO>::kBytes;
  static constexpr int T = 32 / ESZ;        // positions per lane: 16 bf16 / 8 fp32 (32 bytes)
  static constexpr int TB = 16 / ESZ;       // positions per 16-byte vector
  static constexpr int LCH = 32 * T;        // positions per chunk
  static constexpr int SMEM = 2 * 2 * N * LCH * ESZ;  // two buffers of the B and C tiles
};

// T io values starting at position l of a row (row_base points at position 0)
template <typename IO, typename Cfg>
__device__ __forceinline__ void load_run(const IO* row_base, int64_t l, int seqlen, float* out) {
  constexpr int T = Cfg::T, TB = Cfg::TB;
  if constexpr (Cfg::VEC) {
#pragma unroll
    for (int v = 0; v < T / TB; ++v) {
      const int64_t lv = l + v * TB;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (lv < seqlen) w = __ldg(reinterpret_cast<const uint4*>(row_base + lv));
      if constexpr (sizeof(IO) == 2) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          out[v * TB + 2 * k] = bf16lo(ws[k]);
          out[v * TB + 2 * k + 1] = bf16hi(ws[k]);
        }
      } else {
        out[v * TB + 0] = __uint_as_float(w.x);
        out[v * TB + 1] = __uint_as_float(w.y);
        out[v * TB + 2] = __uint_as_float(w.z);
        out[v * TB + 3] = __uint_as_float(w.w);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < T; ++i) out[i] = (l + i < seqlen) ? Io<IO>::ldg(row_base + l + i) : 0.0f;
  }
}

template <typename IO, typename Cfg>
__device__ __forceinline__ void store_run(IO* row_base, int64_t l, int seqlen, const float* v) {
  constexpr int T = Cfg::T, TB = Cfg::TB;
  if constexpr (Cfg::VEC) {
#pragma unroll
    for (int q = 0; q < T / TB; ++q) {
      const int64_t lv = l + q * TB;
      if (lv < seqlen) {
        uint4 w;
        if constexpr (sizeof(IO) == 2) {
          w = make_uint4(pack_bf16x2(v[q * TB + 0], v[q * TB + 1]),
                         pack_bf16x2(v[q * TB + 2], v[q * TB + 3]),
                         pack_bf16x2(v[q * TB + 4], v[q * TB + 5]),
                         pack_bf16x2(v[q * TB + 6], v[q * TB + 7]));
        } else {
          w = make_uint4(__float_as_uint(v[q * TB + 0]), __float_as_uint(v[q * TB + 1]),
                         __float_as_uint(v[q * TB + 2]), __float_as_uint(v[q * TB + 3]));
        }
        *reinterpret_cast<uint4*>(row_base + lv) = w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < T; ++i)
      if (l + i < seqlen) Io<IO>::store(row_base + l + i, v[i]);
  }
}

// T io values of a staged [position] run in shared memory into fp32
template <typename IO, int T>
__device__ __forceinline__ void lds_run(const IO* q, float* out) {
#pragma unroll
  for (int v = 0; v < T * static_cast<int>(sizeof(IO)) / 16; ++v) {
    const uint4 w = *reinterpret_cast<const uint4*>(q + v * (16 / sizeof(IO)));
    if constexpr (sizeof(IO) == 2) {
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        out[v * 8 + 2 * k] = bf16lo(ws[k]);
        out[v * 8 + 2 * k + 1] = bf16hi(ws[k]);
      }
    } else {
      out[v * 4 + 0] = __uint_as_float(w.x);
      out[v * 4 + 1] = __uint_as_float(w.y);
      out[v * 4 + 2] = __uint_as_float(w.z);
      out[v * 4 + 3] = __uint_as_float(w.w);
    }
  }
}

// Stage B and C of chunk k of batch row b: tile[t][n][i] = (t ? C : B)[b][n][k*LCH + i],
// zero past the end of the sequence.
template <typename IO, typename Cfg>
__device__ __forceinline__ void chunk_stage_bc(const ScanParams& p, int b, int k, IO* tile) {
  constexpr int N = Cfg::N, LCH = Cfg::LCH;
  const IO* src[2] = {static_cast<const IO*>(p.B) + static_cast<int64_t>(b) * N * p.seqlen,
                      static_cast<const IO*>(p.C) + static_cast<int64_t>(b) * N * p.seqlen};
  const int64_t l0 = static_cast<int64_t>(k) * LCH;
  if constexpr (Cfg::VEC) {
    constexpr int PPV = 16 / static_cast<int>(sizeof(IO));  // positions per 16 bytes
    constexpr int VPR = LCH / PPV;                          // vectors per state row
    for (int c = threadIdx.x; c < 2 * N * VPR; c += Cfg::THREADS) {
      const int v = c % VPR, n = (c / VPR) % N, t = c / (VPR * N);
      const int64_t l = l0 + static_cast<int64_t>(v) * PPV;
      const bool ok = l < p.seqlen;
      const IO* g = (t ? src[1] : src[0]) + (ok ? static_cast<int64_t>(n) * p.seqlen + l : 0);
      cp_async16_zfill(tile + (t * N + n) * LCH + v * PPV, g, ok);
    }
  } else {
    for (int e = threadIdx.x; e < 2 * N * LCH; e += Cfg::THREADS) {
      const int i = e % LCH, n = (e / LCH) % N, t = e / (LCH * N);
      const int64_t l = l0 + i;
      IO v = IO(0);
      if (l < p.seqlen) v = (t ? src[1] : src[0])[static_cast<int64_t>(n) * p.seqlen + l];
      tile[(t * N + n) * LCH + i] = v;
    }
  }
}

// The per-state loop of one chunk for the warp that owns the channel: pairs, warp
// scan, carry and replay with y += C h.  AR: kArFast (1 - Abar) B u / -A, kArNeg the
// accurate coefficient for negative A, kArGen the accurate one for any A.
template <typename IO, typename Cfg, int AR, bool CKPT>
__device__ __forceinline__ void chunk_states(const float* Arow, int lane, const IO* tile,
                                             const float* s, const float* u, float* y,
                                             float* carry, float* ck, int64_t ck_stride,
                                             int64_t l, int seqlen) {
  constexpr bool UACC = AR != kArFast;
  constexpr int N = Cfg::N, T = Cfg::T, LCH = Cfg::LCH;
  const unsigned FULL = 0xffffffffu;
#pragma unroll 2
  for (int n = 0; n < N; ++n) {
    const float An = __ldg(Arow + n);
    const float IAn = (An == 0.0f) ? 0.0f : 1.0f / An;
    const float isZn = (An == 0.0f) ? 1.0f : 0.0f;
    float Bv[T], Cv[T], a[T], bb[T];
    lds_run<IO, T>(tile + n * LCH + lane * T, Bv);
    lds_run<IO, T>(tile + (N + n) * LCH + lane * T, Cv);
    float P = 1.0f, H = 0.0f;
    if constexpr (!Cfg::EULER && (AR == kArFast || AR == kArNeg)) {
      // pairs of positions in packed f32x2 arithmetic (the two ex2 issue in the shadow
      // of the packed FMAs); the fold of H and P stays sequential over the positions
      const f2 An2 = mk2(An, An), nIA2 = mk2(-IAn, -IAn), one = mk2(1.0f, 1.0f);
#pragma unroll
      for (int i = 0; i < T; i += 2) {
        const f2 X = mul2(mk2(Bv[i], Bv[i + 1]), mk2(u[i], u[i + 1]));
        f2 a2, bb2;
        if constexpr (AR == kArFast) {
          const f2 q = mul2(mk2(s[i], s[i + 1]), An2);
          a2 = mk2(ex2(q.x), ex2(q.y));
          bb2 = mul2(mul2(X, nIA2), sub2(one, a2));        // (Abar - 1) B u / A
        } else {
          const f2 nq = mul2(mk2(-s[i], -s[i + 1]), An2);  // -q >= 0
          const f2 ome = one_minus_exp2_neg2(nq, mk2(ex2(-nq.x), ex2(-nq.y)));  // 1 - Abar
          a2 = sub2(one, ome);
          bb2 = mul2(mul2(ome, nIA2), X);                  // (Abar - 1) / A B u
        }
        a[i] = a2.x;
        a[i + 1] = a2.y;
        bb[i] = bb2.x;
        bb[i + 1] = bb2.y;
        H = fmaf(a[i], H, bb[i]);
        P *= a[i];
        H = fmaf(a[i + 1], H, bb[i + 1]);
        P *= a[i + 1];
      }
    } else {
#pragma unroll
    for (int i = 0; i < T; ++i) {
      const float q = s[i] * An;
      const float ahw = ex2(q);
      const float X = Bv[i] * u[i];
      if constexpr (Cfg::EULER) {
        a[i] = UACC ? ((fabsf(q) < kExpm1SeriesMaxQ) ? 1.0f + exp2m1_accurate(q, ahw) : ahw)
                    : ahw;
        bb[i] = (s[i] * kLn2) * X;         // dt B u
      } else if constexpr (!UACC) {
        const float nK = X * (-IAn);       // -B u / A
        a[i] = ahw;
        bb[i] = fmaf(-ahw, nK, nK);        // (Abar - 1) B u / A
      } else if constexpr (AR == kArNeg) {
        const float em1 = exp2m1_neg(q, ahw);
        a[i] = 1.0f + em1;
        bb[i] = (em1 * IAn) * X;           // (Abar - 1) / A B u
      } else {
        const float em1 = exp2m1_accurate(q, ahw);
        a[i] = (fabsf(q) < kExpm1SeriesMaxQ) ? 1.0f + em1 : ahw;
        const float coef = fmaf(isZn, s[i] * kLn2, em1 * IAn);
        bb[i] = coef * X;
      }
      H = fmaf(a[i], H, bb[i]);
      P *= a[i];
    }
    }
    // inclusive warp scan of (P, H) over lanes (lane order = position order)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float Pu = __shfl_up_sync(FULL, P, o);
      const float Hu = __shfl_up_sync(FULL, H, o);
      if (lane >= o) {
        H = fmaf(P, Hu, H);
        P *= Pu;
      }
    }
    const float Pe = __shfl_up_sync(FULL, P, 1);
    const float He = __shfl_up_sync(FULL, H, 1);
    const float P31 = __shfl_sync(FULL, P, 31);
    const float H31 = __shfl_sync(FULL, H, 31);
    const float cin = carry[n];
    float hs = (lane == 0) ? cin : fmaf(Pe, cin, He);
    __syncwarp();
    if (lane == 0) carry[n] = fmaf(P31, cin, H31);
    // training forward: the states entering this lane's checkpoint blocks (its first
    // position, and position 8 of 16); a lane's row of a checkpoint is written state by
    // state and merges in L2
    if (CKPT && l < seqlen) ck[(l / kCkptPos) * ck_stride + n] = hs;
#pragma unroll
    for (int i = 0; i < T; ++i) {
      hs = fmaf(a[i], hs, bb[i]);
      y[i] = fmaf(Cv[i], hs, y[i]);
      if constexpr (T > kCkptPos) {
        if (CKPT && i % kCkptPos == kCkptPos - 1 && i + 1 < T && l + i + 1 < seqlen)
          ck[((l + i + 1) / kCkptPos) * ck_stride + n] = hs;
      }
    }
  }
}

// One chunk of one channel for the warp that owns it; `carry` ([N], this warp's,
// in shared memory) holds the state entering the chunk and receives the state after
// it; `tile` holds the chunk's B and C.  ACC: accurate arithmetic throughout (fp32
// io, or small |A|); otherwise a chunk holding a step with |q| = s |A| below
// kFastPathMinQ (s_min = kFastPathMinQ / min |A|) takes the accurate update.
template <typename IO, typename Cfg, bool ACC, bool CKPT>
__device__ __forceinline__ void chunk_channel(const ScanParams& p, int b, int d, int lane, int k,
                                              const IO* tile, float* carry, float s_min,
                                              bool neg) {
  constexpr int T = Cfg::T, LCH = Cfg::LCH;
  const int64_t row = static_cast<int64_t>(b) * p.dim + d;
  const IO* urow = static_cast<const IO*>(p.u) + row * p.seqlen;
  const IO* drow = static_cast<const IO*>(p.delta) + row * p.seqlen;
  const IO* zrow = Cfg::GATE ? static_cast<const IO*>(p.z) + row * p.seqlen : nullptr;
  IO* yrow = static_cast<IO*>(p.y) + row * p.seqlen;
  const float* Arow = p.A + static_cast<int64_t>(d) * Cfg::N;
  const float Dd = p.D ? __ldg(p.D + d) : 0.0f;
  const float bias2 = p.bias ? __ldg(p.bias + d) * kLog2e : 0.0f;

  const int64_t l = static_cast<int64_t>(k) * LCH + lane * T;  // this lane's first position
  float s[T], u[T], y[T];
  load_run<IO, Cfg>(urow, l, p.seqlen, u);
  load_run<IO, Cfg>(drow, l, p.seqlen, s);
  bool slow = false;
#pragma unroll
  for (int i = 0; i < T; ++i) {
    const float x2 = fmaf(s[i], kLog2e, bias2);
    const float sv = p.softplus ? (ACC ? softplus_log2_accurate(x2) : softplus_log2_fast(x2)) : x2;
    const bool in = l + i < p.seqlen;
    s[i] = in ? sv : 0.0f;  // past the end: identity pair (1, 0)
    slow |= in && !(sv >= s_min);
    y[i] = 0.0f;
  }
  float* const ck = CKPT ? p.ckpt + row * Cfg::N : nullptr;
  const int64_t ck_stride = static_cast<int64_t>(p.batch) * p.dim * Cfg::N;
  if constexpr (Cfg::EULER) {
    // (the Euler input term dt B u has no cancellation at small steps)
    chunk_states<IO, Cfg, ACC ? kArGen : kArFast, CKPT>(Arow, lane, tile, s, u, y, carry, ck,
                                                  ck_stride, l, p.seqlen);
  } else {
    if (!ACC && !__any_sync(0xffffffffu, slow))
      chunk_states<IO, Cfg, kArFast, CKPT>(Arow, lane, tile, s, u, y, carry, ck, ck_stride, l,
                                     p.seqlen);
    else if (neg)
      chunk_states<IO, Cfg, kArNeg, CKPT>(Arow, lane, tile, s, u, y, carry, ck, ck_stride, l,
                                    p.seqlen);
    else
      chunk_states<IO, Cfg, kArGen, CKPT>(Arow, lane, tile, s, u, y, carry, ck, ck_stride, l,
                                    p.seqlen);
  }
  float z[T];
  if constexpr (Cfg::GATE) load_run<IO, Cfg>(zrow, l, p.seqlen, z);
#pragma unroll
  for (int i = 0; i < T; ++i) {
    float v = fmaf(Dd, u[i], y[i]);
    if constexpr (Cfg::GATE) v *= (ACC ? silu_accurate(z[i]) : silu_fast(z[i]));
    y[i] = v;
  }
  store_run<IO, Cfg>(yrow, l, p.seqlen, y);
  __syncwarp();
}

// Grid: x = batch row * ceil(dim / WARPS) + channel group; warp w of a CTA owns
// channel group * WARPS + w of that batch row (warps past dim only stage).
// CKPT: the training forward (state checkpoints to p.ckpt), compiled apart
template <typename IO, typename Cfg, bool CKPT = false>
__global__ void __launch_bounds__(Cfg::THREADS) scan_chunk_kernel(const ScanParams p) {
  extern __shared__ __align__(16) unsigned char chunk_smem[];
  __shared__ float carry_smem[Cfg::WARPS][Cfg::N];
  constexpr int N = Cfg::N, LCH = Cfg::LCH;
  IO* tiles = reinterpret_cast<IO*>(chunk_smem);  // 2 buffers of [2][N][LCH]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* carry = carry_smem[warp];
  const int groups = (p.dim + Cfg::WARPS - 1) / Cfg::WARPS;
  const int b = static_cast<int>(blockIdx.x / groups);
  const int d = static_cast<int>(blockIdx.x % groups) * Cfg::WARPS + warp;
  const bool active = d < p.dim;
  const int64_t row = static_cast<int64_t>(b) * p.dim + d;

  // fast or accurate arithmetic per warp (bf16 io with every |A| >= the fast-path bound)
  bool acc = true;
  if constexpr (sizeof(IO) == 2) {
    bool small_a = false;
    if (active)
      for (int n = lane; n < N; n += 32)
        small_a |= !(fabsf(__ldg(p.A + static_cast<int64_t>(d) * N + n)) >= kFastPathMinAbsA);
    acc = __any_sync(0xffffffffu, small_a);
  }
  // every A of the channel negative: the accurate update needs no branch
  bool neg = true;
  if (active)
    for (int n = lane; n < N; n += 32) neg = neg && __ldg(p.A + static_cast<int64_t>(d) * N + n) < 0.0f;
  neg = __all_sync(0xffffffffu, neg);
  // smallest step size (log2 units) the fast update takes for this channel
  float s_min = 0.0f;
  if (sizeof(IO) == 2 && !acc && active) {
    float amin = fabsf(__ldg(p.A + static_cast<int64_t>(d) * N));
    for (int n = 1; n < N; ++n) amin = fminf(amin, fabsf(__ldg(p.A + static_cast<int64_t>(d) * N + n)));
    s_min = kFastPathMinQ / amin;
  }
  if (active && lane < N) carry[lane] = p.h0 ? __ldg(p.h0 + row * N + lane) : 0.0f;

  const int nch = (p.seqlen + LCH - 1) / LCH;
  chunk_stage_bc<IO, Cfg>(p, b, 0, tiles);
  cp_async_commit();
#pragma unroll 1
  for (int k = 0; k < nch; ++k) {
    IO* cur = tiles + (k & 1) * 2 * N * LCH;
    cp_async_wait_all();
    __syncthreads();  // chunk k's B and C visible; chunk k - 1's buffer free
    if (k + 1 < nch) {
      chunk_stage_bc<IO, Cfg>(p, b, k + 1, tiles + ((k + 1) & 1) * 2 * N * LCH);
      cp_async_commit();
    }
    if (active) {
      if (acc)
        chunk_channel<IO, Cfg, true, CKPT>(p, b, d, lane, k, cur, carry, s_min, neg);
      else
        chunk_channel<IO, Cfg, false, CKPT>(p, b, d, lane, k, cur, carry, s_min, neg);
    }
  }
  if (active && p.h_last && lane < N) p.h_last[row * N + lane] = carry[lane];
}

}  // namespace ssm
