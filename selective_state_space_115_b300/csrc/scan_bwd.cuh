// scan_bwd.cuh -- gradient of the selective scan (reverse mode), for training.
//
// Mamba_Model_Report.md, section 4.1, differentiates the recurrence
// H[t] = A[t] H[t-1] + X[t] with a reverse scan (pscan_rev): the adjoint
// g_l = dLoss/dh_l runs from the end, g_{l-1} = Abar_l g_l + (terms of l-1), and
// each position's partials follow from g_l and the state before it.  With the
// ZOH step h_l = Abar h_{l-1} + coef B u (Abar = exp(dt A), coef = expm1(dt A)/A)
// the partials per (channel, position, state) are
//
//   dC  += dy0 h_l                 dB += g coef u          du += g coef B
//   ddt += Abar g (A h_{l-1} + B u)                   (Euler: A Abar g h_{l-1} + g B u)
//   dA  += g (dt Abar h_{l-1} + dcoef/dA B u)         (Euler: dcoef/dA = 0)
//
// with dy0 the gradient of the output before the silu gate, and ddelta = ddt *
// sigmoid(delta + bias) through the softplus.  "Mamba学习记录" (lengnian), Part3,
// names recomputation among the hardware-aware algorithm's means of keeping
// intermediate results cheap: the states are not stored by the forward pass but
// recomputed here.
//
// Layout and schedule (one CTA = THREADS/4 channels of one batch row, four lanes
// per channel, each lane owning N/4 states):
//   phase 1  forward over the whole sequence, writing the state entering every
//            block of kBwdPos (8) positions to a workspace checkpoint
//            [block][row][N];
//   phase 2  blocks in reverse: recompute the block's states per lane into
//            registers from its checkpoint (8 positions x N/4 states), then run
//            the adjoint backwards through the block.
// Eight-position blocks keep the trajectory at 32 registers, so four CTAs of 128
// threads fit an SM (at 16 positions three did); the checkpoints take 4 bytes
// per state every 8 positions, written once and read once.
// u, delta, z, dy stream through a two-stage shared-memory ring filled by
// cp.async; B and C are prefetched into registers one block ahead and parked in
// shared memory as fp32 [position][state].  dB and dC are sums over the channels:
// each warp reduce-scatters its 8 channels with shuffles, the CTA sums its warps
// through shared memory and writes one partial per (CTA, batch row, state,
// position); a second kernel adds the partials of a batch row in a fixed order,
// so the result does not depend on scheduling.  dA, dD and the bias gradient are
// per-channel sums over positions, added over the batch rows by that kernel.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

constexpr int kBwdPos = 8;  // positions per block = checkpoint stride
constexpr int kBwdLpc = 4;   // lanes per channel
constexpr int kBwdPpl = kBwdPos / kBwdLpc;  // positions per lane in the per-position steps

struct BwdParams {
  int64_t batch;
  int dim, seqlen, nblk, tiles;  // tiles: CTAs per batch row
  int softplus;
  const void* u;
  const void* delta;
  const void* z;
  const void* dy;
  const void* B;
  const void* C;
  const float* A;
  const float* D;
  const float* bias;
  const float* h0;
  const float* dh_last;
  void* du;
  void* ddelta;
  void* dz;
  float* dh0;
  float* ckpt;     // [nblk][batch * dim][N]: state entering each block
  float* part_bc;  // [tiles][batch][2][N][seqlen]: per-CTA partial dB (0), dC (1)
  float* part_a;   // [nseg][batch * dim][N]: per-channel dA of each segment
  float* part_dd;  // [nseg][batch * dim][2]: per-channel dD, bias gradient of each segment
  // sequence split (nseg == 1: none; seg_len = seqlen), segments of seg_len
  // positions (a multiple of kBwdPos); per (segment, channel) from the first pass:
  int nseg, seg_len;
  float* seg_E;    // [nseg][batch * dim][N]: state after the segment from a zero state
  float* seg_R;    // [nseg][batch * dim][N]: the segment's own adjoint at the position before it
  float* seg_sum;  // [nseg][batch * dim]: sum of the segment's step sizes (log2 units)
  // [nseg * batch * tiles] (bf16 ZOH): 1 where the CTA takes the fast coefficients
  const unsigned char* cta_fast;
  // the training forward's checkpoints, [nblk][batch * dim][N] in state order (the
  // state entering every block): when given, the gradient runs no forward pass of its
  // own (phase 1 and the segments' forward half are skipped)
  const float* ckpt_in;
};

template <typename IO, int N_, bool GATE_, bool EULER_, bool VEC_, int THREADS_ = 128>
struct BwdCfg {
  using io_t = IO;
  static constexpr int N = N_, NS = N_ / kBwdLpc;
  static constexpr bool GATE = GATE_, EULER = EULER_;
  static constexpr bool VEC = VEC_;  // 16-byte aligned rows: cp.async staging, vector stores
  static constexpr int THREADS = THREADS_, WARPS = THREADS_ / 32, CH = THREADS_ / kBwdLpc;
  static constexpr int ES = sizeof(IO);
  static constexpr int ROWB = kBwdPos * ES;  // one channel's block row (bytes)
  static constexpr int CHB = CH * ROWB;      // one per-channel tile: [CH][16]
  static constexpr int STAGE = 4 * CHB;      // u, delta, z, dy
  static constexpr int BCS = N + 4;          // row of the fp32 B / C tile (padded)
  // B and C are parked once per lane state order (NS orders, see bwd_perm)
  static constexpr int BCB = 2 * NS * kBwdPos * BCS * 4;
  static constexpr int SCS = kBwdPos + 4;    // per-channel row of S / SG / DY0 (padded)
  static constexpr int REDS = kBwdPos * 8 + 4;  // per-channel stride of RED (padded)
  static constexpr int WBS = kBwdPos + 1;       // position row of WB (padded)
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_BC = OFF_STAGE + 2 * STAGE;
  static constexpr int OFF_S = OFF_BC + 2 * BCB;
  static constexpr int OFF_SG = OFF_S + CH * SCS * 4;
  static constexpr int OFF_DY0 = OFF_SG + CH * SCS * 4;
  static constexpr int OFF_RED = OFF_DY0 + CH * SCS * 4;
  static constexpr int OFF_WB = OFF_RED + CH * REDS * 4;
  static constexpr int OFF_OUT = OFF_WB + WARPS * 2 * N * WBS * 4;
  static constexpr int SMEM = OFF_OUT + 3 * CHB;
  static_assert(N % kBwdLpc == 0 && NS >= 1 && NS <= 4, "dstate 4, 8 or 16");
  static constexpr int BC_EPT = (N * kBwdPos + THREADS - 1) / THREADS;  // B/C elements per thread
  static_assert(OFF_BC % 16 == 0 && OFF_S % 16 == 0 && OFF_RED % 16 == 0 && OFF_OUT % 16 == 0,
                "16-byte aligned regions");
};

// 2^x on the special-function unit, as an asm statement the compiler may not
// merge with an identical one: the adjoint recomputes Abar rather than holding
// the forward recompute's 16 x NS values in registers across the two passes
__device__ __forceinline__ float ex2_fresh(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// d coef / d A of the ZOH coefficient coef = (e^{dt A} - 1) / A, with q = dt A
// log2(e): the difference (dt Abar - coef) / A cancels for small |q|, where the
// Taylor series dt^2 (1/2 + x/3 + x^2/8 + x^3/30 + x^4/144) (x = dt A) is used
// instead (truncation below 2e-8 relative for |q| < 1/8); at A = 0 it gives the
// limit dt^2 / 2.  SHORT (the fast coefficients of bf16 io) keeps three terms,
// written in q: truncation below (x^3 / 30) / (1/2) < 4.4e-5 relative for |q| < 1/8,
// under the direct form's own error there (its coefficient carries the hardware
// ex2's ~2^-22, which the cancellation raises to ~2^-21 / x^2 = 6e-5).
template <bool SHORT>
__device__ __forceinline__ float dcoef_dA(float dt, float q, float ra, float abar, float coef) {
  float ps;
  if constexpr (SHORT) {
    // 1/2 + (ln2 / 3) q + (ln2^2 / 8) q^2
    ps = fmaf(fmaf(q, 0.06005662673977513f, 0.23104906018664842f), q, 0.5f);
  } else {
    const float x = q * kLn2;
    ps = fmaf(x, 1.0f / 144.0f, 1.0f / 30.0f);
    ps = fmaf(ps, x, 0.125f);
    ps = fmaf(ps, x, 1.0f / 3.0f);
    ps = fmaf(ps, x, 0.5f);
  }
  const float series = (dt * dt) * ps;
  const float direct = fmaf(dt, abar, -coef) * ra;
  return (fabsf(q) < kExpm1SeriesMaxQ) ? series : direct;
}

// dcoef_dA<true> for a pair of states in packed f32x2 (the same operations, so the
// same bits); `ncoef` is -coef, exactly
__device__ __forceinline__ f2 dcoef_dA_short2(f2 dtsq, f2 dt, f2 q, f2 ra, f2 abar, f2 ncoef) {
  const f2 ps = fma2(fma2(q, mk2(0.06005662673977513f, 0.06005662673977513f),
                          mk2(0.23104906018664842f, 0.23104906018664842f)),
                     q, mk2(0.5f, 0.5f));
  const f2 series = mul2(dtsq, ps);
  const f2 direct = mul2(fma2(dt, abar, ncoef), ra);
  return mk2((fabsf(q.x) < kExpm1SeriesMaxQ) ? series.x : direct.x,
             (fabsf(q.y) < kExpm1SeriesMaxQ) ? series.y : direct.y);
}

// the ZOH (or Euler) input coefficient for one state: FAST takes Abar - 1
// directly (bf16 io with |A| >= 1/8, as the forward's fast path), otherwise the
// expm1 series near zero and the dt limit at A = 0
template <bool EULER, bool FAST>
__device__ __forceinline__ float bwd_coef(float q, float dt, float a, float ra, float abar) {
  if constexpr (EULER) {
    return dt;
  } else if constexpr (FAST) {
    return fmaf(abar, ra, -ra);
  } else {
    const float em1 = exp2m1_accurate(q, abar);
    return (a == 0.0f) ? dt : em1 * ra;
  }
}

// Lane state order.  Lane `part` of a channel owns states n0 .. n0+NS-1 (n0 =
// part*NS), held in slot order: slot k is state n0 + (k ^ perm), with perm taken
// from the lane bits that the channel reduction below pairs over (bits 4, 3 of
// the lane).  The order makes that reduction's exchanges the same for every lane.
template <int NS>
__device__ __forceinline__ int bwd_perm(int lane) {
  return NS == 4 ? (lane >> 3) & 3 : NS == 2 ? (lane >> 4) & 1 : 0;
}

// Warp reduce-scatter over the 8 channels of a warp (lane bits 2..4): v holds
// this lane's NS slots of one channel; returns the sum over the warp's channels
// of state n0 + bwd_perm(lane), which lanes with bwd_rs_holder(lane) hold once.
// In slot order the partner of every exchange keeps the slots this lane sends,
// so no lane-dependent selection is needed.
template <int NS>
__device__ __forceinline__ float bwd_rs(const float (&v)[NS]) {
  constexpr unsigned kAll = 0xffffffffu;
  if constexpr (NS == 4) {
    const float k0 = v[0] + __shfl_xor_sync(kAll, v[2], 16);
    const float k1 = v[1] + __shfl_xor_sync(kAll, v[3], 16);
    float x = k0 + __shfl_xor_sync(kAll, k1, 8);
    x += __shfl_xor_sync(kAll, x, 4);
    return x;
  } else if constexpr (NS == 2) {
    float x = v[0] + __shfl_xor_sync(kAll, v[1], 16);
    x += __shfl_xor_sync(kAll, x, 8);
    x += __shfl_xor_sync(kAll, x, 4);
    return x;
  } else {
    float x = v[0];
    x += __shfl_xor_sync(kAll, x, 16);
    x += __shfl_xor_sync(kAll, x, 8);
    x += __shfl_xor_sync(kAll, x, 4);
    return x;
  }
}
template <int NS>
__device__ __forceinline__ bool bwd_rs_holder(int lane) {
  return (lane & (NS == 4 ? 4 : NS == 2 ? 12 : 28)) == 0;
}

// Stage the per-channel tiles (u, delta and, when `full`, z and dy) of positions
// l0 .. l0+kBwdPos-1 of the CTA's channels; positions past the end and channels past
// dim read as zero.
template <typename Cfg>
__device__ __forceinline__ void bwd_stage(const BwdParams& p, unsigned char* st, int64_t rowbase,
                                          int d0, int l0, bool full) {
  using IO = typename Cfg::io_t;
  const int ntens = full ? 4 : 2;
  auto src = [&](int t) -> const IO* {
    return static_cast<const IO*>(t == 0 ? p.u : t == 1 ? p.delta : t == 2 ? p.z : p.dy);
  };
  if constexpr (Cfg::VEC) {
    constexpr int CPR = Cfg::ROWB / 16;  // 16-byte chunks per row
    constexpr int PPC = 16 / Cfg::ES;    // positions per chunk
    const int total = ntens * Cfg::CH * CPR;
    for (int c = threadIdx.x; c < total; c += Cfg::THREADS) {
      const int k = c % CPR, ch = (c / CPR) % Cfg::CH, t = c / (CPR * Cfg::CH);
      if (t == 2 && !Cfg::GATE) continue;
      const int d = d0 + ch, l = l0 + k * PPC;
      const bool ok = d < p.dim && l < p.seqlen;
      const IO* g = src(t) +
                    (ok ? (rowbase + d) * static_cast<int64_t>(p.seqlen) + l : 0);
      cp_async16_zfill(st + t * Cfg::CHB + ch * Cfg::ROWB + k * 16, g, ok);
    }
  } else {
    const int total = ntens * Cfg::CH * kBwdPos;
    for (int e = threadIdx.x; e < total; e += Cfg::THREADS) {
      const int pp = e % kBwdPos, ch = (e / kBwdPos) % Cfg::CH, t = e / (kBwdPos * Cfg::CH);
      if (t == 2 && !Cfg::GATE) continue;
      const int d = d0 + ch, l = l0 + pp;
      IO v = IO(0);
      if (d < p.dim && l < p.seqlen)
        v = src(t)[(rowbase + d) * static_cast<int64_t>(p.seqlen) + l];
      reinterpret_cast<IO*>(st + t * Cfg::CHB + ch * Cfg::ROWB)[pp] = v;
    }
  }
}

// B (and C) of positions l0 .. l0+kBwdPos-1 of batch row b: element e = t + i * THREADS
// (state e / 16, position e % 16) goes to thread t's register i as raw io bits;
// bwd_bc_park converts and stores them as fp32 [order][position][state], once in
// each lane state order (B: orders 0 .. NS-1, then C).
template <typename Cfg>
__device__ __forceinline__ void bwd_bc_fetch(const BwdParams& p, int64_t b, int l0, bool withC,
                                             typename Cfg::io_t (&rb)[Cfg::BC_EPT],
                                             typename Cfg::io_t (&rc)[Cfg::BC_EPT]) {
  using IO = typename Cfg::io_t;
#pragma unroll
  for (int i = 0; i < Cfg::BC_EPT; ++i) {
    rb[i] = IO(0);
    rc[i] = IO(0);
    const int e = threadIdx.x + i * Cfg::THREADS;
    if (e < Cfg::N * kBwdPos) {
      const int n = e / kBwdPos, l = l0 + e % kBwdPos;
      if (l < p.seqlen) {
        const int64_t off = (b * Cfg::N + n) * static_cast<int64_t>(p.seqlen) + l;
        rb[i] = static_cast<const IO*>(p.B)[off];
        if (withC) rc[i] = static_cast<const IO*>(p.C)[off];
      }
    }
  }
}
template <typename Cfg>
__device__ __forceinline__ void bwd_bc_park(float* bc, const typename Cfg::io_t (&rb)[Cfg::BC_EPT],
                                            const typename Cfg::io_t (&rc)[Cfg::BC_EPT]) {
  using IO = typename Cfg::io_t;
#pragma unroll
  for (int i = 0; i < Cfg::BC_EPT; ++i) {
    const int e = threadIdx.x + i * Cfg::THREADS;
    if (e < Cfg::N * kBwdPos) {
      const int n = e / kBwdPos, pp = e % kBwdPos;
      const float vb = Io<IO>::load(&rb[i]), vc = Io<IO>::load(&rc[i]);
      constexpr int NS = Cfg::NS;
#pragma unroll
      for (int c = 0; c < NS; ++c) {  // order c: state n at slot (n ^ c) within its group
        const int col = (n & ~(NS - 1)) | ((n & (NS - 1)) ^ c);
        bc[(c * kBwdPos + pp) * Cfg::BCS + col] = vb;
        bc[((NS + c) * kBwdPos + pp) * Cfg::BCS + col] = vc;
      }
    }
  }
}

// this lane's NS consecutive states of a [position][state] fp32 row (16-byte
// aligned for NS = 4, 8-byte for NS = 2)
template <int NS>
__device__ __forceinline__ void ld_states(const float* q, float (&v)[NS]) {
  if constexpr (NS == 4) {
    const float4 t = *reinterpret_cast<const float4*>(q);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (NS == 2) {
    const float2 t = *reinterpret_cast<const float2*>(q);
    v[0] = t.x; v[1] = t.y;
  } else {
    v[0] = q[0];
  }
}

template <typename IO>
__device__ __forceinline__ float ld_io(const unsigned char* tile, int ch_rowb, int pp) {
  return Io<IO>::load(reinterpret_cast<const IO*>(tile + ch_rowb) + pp);
}

// step size in log2 units, s = dt * log2(e), and sigmoid(delta + bias), for this
// lane's positions part*kBwdPpl .. (part+1)*kBwdPpl-1 of its channel
template <typename Cfg>
__device__ __forceinline__ void bwd_prologue(const BwdParams& p, const unsigned char* stage,
                                             int chl, int part, float bias, float* S, float* SG,
                                             bool want_sigmoid) {
  using IO = typename Cfg::io_t;
#pragma unroll
  for (int i = 0; i < kBwdPpl; ++i) {
    const int pp = part * kBwdPpl + i;
    const float x = ld_io<IO>(stage + Cfg::CHB, chl * Cfg::ROWB, pp) + bias;
    const float x2 = x * kLog2e;
    float s = x2, sg = 1.0f;
    if (p.softplus) {
      if constexpr (sizeof(IO) == 2) {
        s = softplus_log2_fast(x2);
        sg = rcp(1.0f + ex2(-x2));
      } else {
        s = softplus_log2_accurate(x2);
        sg = 1.0f / (1.0f + expf(-x));
      }
    }
    S[chl * Cfg::SCS + pp] = s;
    if (want_sigmoid) SG[chl * Cfg::SCS + pp] = sg;
  }
}

// phase 1 body for one block: advance this lane's states over the block
template <typename Cfg, bool FAST>
__device__ __forceinline__ void bwd_advance(const BwdParams& p, const unsigned char* stage,
                                            const float* Bt, const float* S, int chl, int n0,
                                            int l0, const float (&a)[Cfg::NS],
                                            const float (&ra)[Cfg::NS], float (&h)[Cfg::NS]) {
  using IO = typename Cfg::io_t;
  constexpr int NS = Cfg::NS;
#pragma unroll
  for (int pp = 0; pp < kBwdPos; ++pp) {
    if (l0 + pp < p.seqlen) {
      const float s = S[chl * Cfg::SCS + pp];
      const float dt = s * kLn2;
      const float uf = ld_io<IO>(stage, chl * Cfg::ROWB, pp);
      float Bv[NS];
      ld_states<NS>(Bt + pp * Cfg::BCS + n0, Bv);
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const float q = s * a[k];
        const float ab = ex2(q);
        const float coef = bwd_coef<Cfg::EULER, FAST>(q, dt, a[k], ra[k], ab);
        h[k] = fmaf(ab, h[k], coef * (Bv[k] * uf));
      }
    }
  }
}

// phase 2 body for one block: recompute the states, then the adjoint backwards
template <typename Cfg, bool FAST>
__device__ __forceinline__ void bwd_block(const BwdParams& p, const unsigned char* stage,
                                          const float* Bt, const float* Ct, const float* S,
                                          float* DY0, float* RED,
                                          float* WB, unsigned char* OUT, int chl, int part,
                                          int lane, int warp, int n0, int l0, float Dd,
                                          const float (&a)[Cfg::NS], const float (&ra)[Cfg::NS],
                                          const float (&nra)[Cfg::NS],
                                          const float (&he)[Cfg::NS], float (&g)[Cfg::NS],
                                          float (&an)[Cfg::NS], float (&dA)[Cfg::NS],
                                          float& dD_acc) {
  using IO = typename Cfg::io_t;
  constexpr int NS = Cfg::NS, N = Cfg::N;

  // ---- forward recompute: traj[pp] = h after position pp; this lane's part of
  // the contraction sum_n C h goes to RED (the du slot, free until the adjoint)
  float traj[kBwdPos][NS];
  {
    float h[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) h[k] = he[k];
#pragma unroll
    for (int pp = 0; pp < kBwdPos; ++pp) {
      if (l0 + pp < p.seqlen) {
        const float s = S[chl * Cfg::SCS + pp];
        const float dt = s * kLn2;
        const float uf = ld_io<IO>(stage, chl * Cfg::ROWB, pp);
        float Bv[NS], Cv[NS];
        ld_states<NS>(Bt + pp * Cfg::BCS + n0, Bv);
        ld_states<NS>(Ct + pp * Cfg::BCS + n0, Cv);
        float y = 0.0f;
        if constexpr (NS % 2 == 0) {
          // state pairs in packed f32x2: the per-state operations of the scalar form
          // below, the contraction summed per pair then across
          const f2 s2 = mk2(s, s), u2 = mk2(uf, uf);
          f2 y2 = mk2(0.0f, 0.0f);
#pragma unroll
          for (int k = 0; k < NS; k += 2) {
            const f2 a2 = mk2(a[k], a[k + 1]);
            const f2 q = mul2(s2, a2);
            const f2 ab = mk2(ex2(q.x), ex2(q.y));
            f2 coef;
            if constexpr (FAST && !Cfg::EULER) {
              coef = fma2(ab, mk2(ra[k], ra[k + 1]), mk2(nra[k], nra[k + 1]));
            } else {
              coef = mk2(bwd_coef<Cfg::EULER, FAST>(q.x, dt, a[k], ra[k], ab.x),
                         bwd_coef<Cfg::EULER, FAST>(q.y, dt, a[k + 1], ra[k + 1], ab.y));
            }
            const f2 hn = fma2(ab, mk2(h[k], h[k + 1]),
                               mul2(coef, mul2(mk2(Bv[k], Bv[k + 1]), u2)));
            h[k] = hn.x;
            h[k + 1] = hn.y;
            traj[pp][k] = hn.x;
            traj[pp][k + 1] = hn.y;
            y2 = fma2(mk2(Cv[k], Cv[k + 1]), hn, y2);
          }
          y = y2.x + y2.y;
        } else {
#pragma unroll
          for (int k = 0; k < NS; ++k) {
            const float q = s * a[k];
            const float ab = ex2(q);
            const float coef = bwd_coef<Cfg::EULER, FAST>(q, dt, a[k], ra[k], ab);
            h[k] = fmaf(ab, h[k], coef * (Bv[k] * uf));
            traj[pp][k] = h[k];
            y = fmaf(Cv[k], h[k], y);
          }
        }
        RED[chl * Cfg::REDS + pp * 8 + part] = y;
      }
    }
  }
  __syncwarp();
  // ---- output before the gate, and the gate's gradients, for this lane's
  // positions part*kBwdPpl ..: dy0 = dLoss/d(y before the gate), dz
#pragma unroll
  for (int i = 0; i < kBwdPpl; ++i) {
    const int pp = part * kBwdPpl + i;
    if (l0 + pp < p.seqlen) {
      const float4 yp = lds128f(RED + chl * Cfg::REDS + pp * 8);
      const float uf = ld_io<IO>(stage, chl * Cfg::ROWB, pp);
      const float y0 = fmaf(Dd, uf, (yp.x + yp.y) + (yp.z + yp.w));
      const float dyf = ld_io<IO>(stage + 3 * Cfg::CHB, chl * Cfg::ROWB, pp);
      float dy0 = dyf;
      if constexpr (Cfg::GATE) {
        const float zf = ld_io<IO>(stage + 2 * Cfg::CHB, chl * Cfg::ROWB, pp);
        float sg;
        if constexpr (sizeof(IO) == 2)
          sg = rcp(1.0f + ex2(-zf * kLog2e));
        else
          sg = 1.0f / (1.0f + expf(-zf));
        dy0 = dyf * zf * sg;
        const float dzv = dyf * y0 * sg * fmaf(zf, 1.0f - sg, 1.0f);
        Io<IO>::store(reinterpret_cast<IO*>(OUT + 2 * Cfg::CHB + chl * Cfg::ROWB) + pp, dzv);
      }
      DY0[chl * Cfg::SCS + pp] = dy0;
      dD_acc = fmaf(dy0, uf, dD_acc);
    }
  }
  __syncwarp();

  // ---- adjoint, positions in reverse
  // dA accumulates per block as dA1 (the Abar term) and dA2 (the coefficient term)
  float dA1[NS], dA2[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) dA1[k] = dA2[k] = 0.0f;
#pragma unroll
  for (int pp = kBwdPos - 1; pp >= 0; --pp) {
    if (l0 + pp < p.seqlen) {
      const float s = S[chl * Cfg::SCS + pp];
      const float dt = s * kLn2;
      const float uf = ld_io<IO>(stage, chl * Cfg::ROWB, pp);
      const float dy0 = DY0[chl * Cfg::SCS + pp];
      float du_p = 0.0f, ddt_p = 0.0f;
      float dBv[NS], dCv[NS], Bs[NS], Cs[NS];
      ld_states<NS>(Bt + pp * Cfg::BCS + n0, Bs);
      ld_states<NS>(Ct + pp * Cfg::BCS + n0, Cs);
      if constexpr (NS % 2 == 0) {
        // state pairs in packed f32x2: the per-state operations of the scalar form
        // below; du and ddt summed per pair then across
        const f2 s2 = mk2(s, s), dt2 = mk2(dt, dt), u2 = mk2(uf, uf), dy2 = mk2(dy0, dy0);
        const f2 dtsq = mk2(dt * dt, dt * dt);
        f2 du2 = mk2(0.0f, 0.0f), ddt2 = mk2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NS; k += 2) {
          const f2 hp = (pp > 0) ? mk2(traj[pp > 0 ? pp - 1 : 0][k], traj[pp > 0 ? pp - 1 : 0][k + 1])
                                 : mk2(he[k], he[k + 1]);
          const f2 a2 = mk2(a[k], a[k + 1]), ra2 = mk2(ra[k], ra[k + 1]);
          const f2 q = mul2(s2, a2);
          const f2 ab = mk2(ex2_fresh(q.x), ex2_fresh(q.y));
          f2 coef;
          if constexpr (FAST && !Cfg::EULER) {
            coef = fma2(ab, ra2, mk2(nra[k], nra[k + 1]));
          } else {
            coef = mk2(bwd_coef<Cfg::EULER, FAST>(q.x, dt, a[k], ra[k], ab.x),
                       bwd_coef<Cfg::EULER, FAST>(q.y, dt, a[k + 1], ra[k + 1], ab.y));
          }
          const f2 B2 = mk2(Bs[k], Bs[k + 1]);
          const f2 gk = fma2(mk2(g[k], g[k + 1]), mk2(an[k], an[k + 1]),
                             mul2(mk2(Cs[k], Cs[k + 1]), dy2));  // dLoss/dh at this position
          const f2 dC = mul2(dy2, mk2(traj[pp][k], traj[pp][k + 1]));
          const f2 gc = mul2(gk, coef);
          const f2 dB = mul2(gc, u2);
          du2 = fma2(gc, B2, du2);
          const f2 bu = mul2(B2, u2);
          const f2 ga = mul2(gk, ab);
          const f2 gdt = mul2(ga, dt2);
          const f2 d1 = fma2(gdt, hp, mk2(dA1[k], dA1[k + 1]));
          dA1[k] = d1.x;
          dA1[k + 1] = d1.y;
          if constexpr (Cfg::EULER) {
            ddt2 = fma2(mul2(ga, a2), hp, fma2(gk, bu, ddt2));
          } else {
            ddt2 = fma2(ga, fma2(a2, hp, bu), ddt2);
            f2 dc;
            if constexpr (FAST) {
              dc = dcoef_dA_short2(dtsq, dt2, q, ra2, ab,
                                   fma2(ab, mk2(nra[k], nra[k + 1]), ra2));  // -coef
            } else {
              dc = mk2(dcoef_dA<false>(dt, q.x, ra[k], ab.x, coef.x),
                       dcoef_dA<false>(dt, q.y, ra[k + 1], ab.y, coef.y));
            }
            const f2 d2 = fma2(mul2(gk, dc), bu, mk2(dA2[k], dA2[k + 1]));
            dA2[k] = d2.x;
            dA2[k + 1] = d2.y;
          }
          dCv[k] = dC.x;
          dCv[k + 1] = dC.y;
          dBv[k] = dB.x;
          dBv[k + 1] = dB.y;
          g[k] = gk.x;
          g[k + 1] = gk.y;
          an[k] = ab.x;
          an[k + 1] = ab.y;
        }
        du_p = du2.x + du2.y;
        ddt_p = ddt2.x + ddt2.y;
      } else {
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const float hp = (pp > 0) ? traj[pp > 0 ? pp - 1 : 0][k] : he[k];
        const float q = s * a[k];
        const float ab = ex2_fresh(q);
        const float coef = bwd_coef<Cfg::EULER, FAST>(q, dt, a[k], ra[k], ab);
        const float gk = fmaf(g[k], an[k], Cs[k] * dy0);  // dLoss/dh at this position
        dCv[k] = dy0 * traj[pp][k];
        const float gc = gk * coef;
        dBv[k] = gc * uf;
        du_p = fmaf(gc, Bs[k], du_p);
        const float bu = Bs[k] * uf;
        const float ga = gk * ab;
        const float gdt = ga * dt;
        dA1[k] = fmaf(gdt, hp, dA1[k]);
        if constexpr (Cfg::EULER) {
          ddt_p = fmaf(ga * a[k], hp, fmaf(gk, bu, ddt_p));
        } else {
          ddt_p = fmaf(ga, fmaf(a[k], hp, bu), ddt_p);
          // dcoef/dA from its series near zero on the fast path too: the difference
          // (dt Abar - coef) / A cancels like dt^2 while its rounding and the
          // hardware ex2's error stay ~2^-24 |B u / A|, so at small |dt A| it would be
          // lost (its relative error grows like 2^-23 / (dt A)^2)
          dA2[k] = fmaf(gk * dcoef_dA<FAST>(dt, q, ra[k], ab, coef), bu, dA2[k]);
        }
        g[k] = gk;
        an[k] = ab;
      }
      }
      RED[chl * Cfg::REDS + pp * 8 + part] = du_p;
      RED[chl * Cfg::REDS + pp * 8 + 4 + part] = ddt_p;
      const float sb = bwd_rs<NS>(dBv);
      const float sc = bwd_rs<NS>(dCv);
      if (bwd_rs_holder<NS>(lane)) {
        const int n = n0 + bwd_perm<NS>(lane);
        WB[((warp * 2 + 0) * N + n) * Cfg::WBS + pp] = sb;
        WB[((warp * 2 + 1) * N + n) * Cfg::WBS + pp] = sc;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NS; ++k) dA[k] += dA1[k] + dA2[k];
}

// First pass of the segmented gradient (nseg > 1), one CTA per (segment, batch
// row, channel tile): the segment's end state from a zero entering state (E), its
// step-size sum, and the adjoint that its own positions send to the position just
// before it from a zero adjoint at its end (R = Abar_a g_a with g_l = Abar_{l+1}
// g_{l+1} + C_l dy0_l).  dy0 does not depend on the states, so R needs no forward
// pass; with E, R and the sums the second pass gives every segment its true
// entering state and its true adjoint at the end (the recurrence and its adjoint
// are linear, and a segment multiplies both by the product of its Abar factors).
template <typename Cfg, bool FAST>
__device__ __forceinline__ void bwd_segment_pass(
    const BwdParams& p, unsigned char* smem, int seg, int64_t b, int d0, int chl, int part, int n0,
    int perm, bool chv, int64_t row, int64_t rowbase, int64_t rows, int l_begin, int j_begin,
    int j_end, float bias, const float (&a)[Cfg::NS], const float (&ra)[Cfg::NS]) {
  using IO = typename Cfg::io_t;
  constexpr int NS = Cfg::NS, N = Cfg::N;
  unsigned char* stage_base = smem + Cfg::OFF_STAGE;
  float* BC = reinterpret_cast<float*>(smem + Cfg::OFF_BC);
  float* S = reinterpret_cast<float*>(smem + Cfg::OFF_S);
  float* SG = reinterpret_cast<float*>(smem + Cfg::OFF_SG);
  auto stage = [&](int i) { return stage_base + i * Cfg::STAGE; };
  auto bcbuf = [&](int i) { return BC + i * (Cfg::BCB / 4); };
  auto bt = [&](int i) { return bcbuf(i) + perm * kBwdPos * Cfg::BCS; };
  auto ct = [&](int i) { return bcbuf(i) + (NS + perm) * kBwdPos * Cfg::BCS; };
  const int nblk = j_end - j_begin;
  IO rb[Cfg::BC_EPT], rc[Cfg::BC_EPT];
  float ssum = 0.0f;

  // forward from a zero state (every segment but the last; not needed when the
  // training forward's checkpoints give every block's entering state)
  if (seg < p.nseg - 1 && !p.ckpt_in) {
    float h[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) h[k] = 0.0f;
    bwd_stage<Cfg>(p, stage(0), rowbase, d0, l_begin, false);
    cp_async_commit();
    bwd_bc_fetch<Cfg>(p, b, l_begin, false, rb, rc);
    bwd_bc_park<Cfg>(bcbuf(0), rb, rc);
    for (int jj = 0; jj < nblk; ++jj) {
      const int l0 = (j_begin + jj) * kBwdPos, buf = jj & 1;
      cp_async_wait_all();
      __syncthreads();
      const bool more = jj + 1 < nblk;
      if (more) {
        bwd_stage<Cfg>(p, stage(buf ^ 1), rowbase, d0, l0 + kBwdPos, false);
        cp_async_commit();
        bwd_bc_fetch<Cfg>(p, b, l0 + kBwdPos, false, rb, rc);
      }
      bwd_prologue<Cfg>(p, stage(buf), chl, part, bias, S, SG, false);
      __syncwarp();
#pragma unroll
      for (int pp = 0; pp < kBwdPos; ++pp)
        if (l0 + pp < p.seqlen) ssum += S[chl * Cfg::SCS + pp];
      bwd_advance<Cfg, FAST>(p, stage(buf), bt(buf), S, chl, n0, l0, a, ra, h);
      if (more) bwd_bc_park<Cfg>(bcbuf(buf ^ 1), rb, rc);
    }
    if (chv) {
#pragma unroll
      for (int k = 0; k < NS; ++k) p.seg_E[(seg * rows + row) * N + n0 + (k ^ perm)] = h[k];
    }
    __syncthreads();  // the stages are reused below
  }

  // adjoint from a zero adjoint at the segment's end (every segment but the first)
  if (seg > 0) {
    float g[NS], an[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      g[k] = 0.0f;
      an[k] = 1.0f;
    }
    const int l_last = (j_end - 1) * kBwdPos;
    bwd_stage<Cfg>(p, stage(0), rowbase, d0, l_last, true);
    cp_async_commit();
    bwd_bc_fetch<Cfg>(p, b, l_last, true, rb, rc);
    bwd_bc_park<Cfg>(bcbuf(0), rb, rc);
    for (int it = 0; it < nblk; ++it) {
      const int j = j_end - 1 - it, l0 = j * kBwdPos, buf = it & 1;
      cp_async_wait_all();
      __syncthreads();
      const bool more = j > j_begin;
      if (more) {
        bwd_stage<Cfg>(p, stage(buf ^ 1), rowbase, d0, l0 - kBwdPos, true);
        cp_async_commit();
        bwd_bc_fetch<Cfg>(p, b, l0 - kBwdPos, true, rb, rc);
      }
      bwd_prologue<Cfg>(p, stage(buf), chl, part, bias, S, SG, false);
      __syncwarp();
      const float* Ct = ct(buf);
#pragma unroll
      for (int pp = kBwdPos - 1; pp >= 0; --pp) {
        if (l0 + pp < p.seqlen) {
          const float s = S[chl * Cfg::SCS + pp];
          if (seg == p.nseg - 1 || p.ckpt_in) ssum += s;
          float dy0 = ld_io<IO>(stage(buf) + 3 * Cfg::CHB, chl * Cfg::ROWB, pp);
          if constexpr (Cfg::GATE) {
            const float zf = ld_io<IO>(stage(buf) + 2 * Cfg::CHB, chl * Cfg::ROWB, pp);
            float sg;
            if constexpr (sizeof(IO) == 2)
              sg = rcp(1.0f + ex2(-zf * kLog2e));
            else
              sg = 1.0f / (1.0f + expf(-zf));
            dy0 = dy0 * zf * sg;
          }
          float Cs[NS];
          ld_states<NS>(Ct + pp * Cfg::BCS + n0, Cs);
#pragma unroll
          for (int k = 0; k < NS; ++k) {
            g[k] = fmaf(g[k], an[k], Cs[k] * dy0);
            an[k] = ex2(s * a[k]);
          }
        }
      }
      if (more) bwd_bc_park<Cfg>(bcbuf(buf ^ 1), rb, rc);
    }
    if (chv) {
#pragma unroll
      for (int k = 0; k < NS; ++k)
        p.seg_R[(seg * rows + row) * N + n0 + (k ^ perm)] = an[k] * g[k];
    }
  }
  if (chv && part == 0) p.seg_sum[seg * rows + row] = ssum;
}

// MODE 0: every CTA, accurate arithmetic (fp32 io, or the Euler term, which needs
// no expm1).  For bf16 io with the ZOH term the work is split over two launches
// compiled separately so that the common case is not held to the register
// budget of the rare one: MODE 1 takes the CTAs whose channels all have
// |A| >= 1/8 (coefficients from Abar - 1, as the forward's fast path), MODE 2
// the others (the series near zero); each returns at once from the CTAs of the other.
constexpr int kBwdAll = 0, kBwdFastTiles = 1, kBwdAccurateTiles = 2;

template <typename Cfg, int MODE, bool PRE>
__global__ void __launch_bounds__(Cfg::THREADS, 4) scan_bwd_kernel(const BwdParams p) {
  constexpr bool FAST = MODE == kBwdFastTiles;
  using IO = typename Cfg::io_t;
  constexpr int NS = Cfg::NS, N = Cfg::N, CH = Cfg::CH;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, part = lane & 3;
  const int chl = tid >> 2;  // channel within the CTA
  // CTA = (segment, batch row, channel tile)
  const int64_t per_seg = p.batch * p.tiles;
  const int seg = static_cast<int>(blockIdx.x / per_seg);
  const int64_t b = (blockIdx.x % per_seg) / p.tiles;
  const int tile = static_cast<int>(blockIdx.x % p.tiles);
  const int d0 = tile * CH;
  const int l_begin = seg * p.seg_len;
  const int l_end = (p.seqlen - l_begin < p.seg_len) ? p.seqlen : l_begin + p.seg_len;
  const int j_begin = l_begin / kBwdPos, j_end = (l_end + kBwdPos - 1) / kBwdPos;
  const int d = d0 + chl;
  const bool chv = d < p.dim;
  const int dc = chv ? d : p.dim - 1;  // clamped for parameter reads
  const int64_t rowbase = b * p.dim;
  const int64_t row = rowbase + dc;
  const int64_t rows = p.batch * p.dim;
  const int n0 = part * NS;
  const int perm = bwd_perm<NS>(lane);  // slot k holds state n0 + (k ^ perm)

  unsigned char* stage_base = smem + Cfg::OFF_STAGE;
  float* BC = reinterpret_cast<float*>(smem + Cfg::OFF_BC);
  float* S = reinterpret_cast<float*>(smem + Cfg::OFF_S);
  float* SG = reinterpret_cast<float*>(smem + Cfg::OFF_SG);
  float* DY0 = reinterpret_cast<float*>(smem + Cfg::OFF_DY0);
  float* RED = reinterpret_cast<float*>(smem + Cfg::OFF_RED);
  float* WB = reinterpret_cast<float*>(smem + Cfg::OFF_WB);
  unsigned char* OUT = smem + Cfg::OFF_OUT;
  auto stage = [&](int i) { return stage_base + i * Cfg::STAGE; };
  auto bcbuf = [&](int i) { return BC + i * (Cfg::BCB / 4); };
  // this lane's order of the parked B and C tiles
  auto bt = [&](int i) { return bcbuf(i) + perm * kBwdPos * Cfg::BCS; };
  auto ct = [&](int i) { return bcbuf(i) + (NS + perm) * kBwdPos * Cfg::BCS; };

  if constexpr (MODE != kBwdAll) {
    // the accurate launch runs first and lets the fast launch start at once (they write
    // disjoint CTAs' outputs); the fast launch's block 0 waits for it before exiting
    if constexpr (MODE == kBwdAccurateTiles) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((p.cta_fast[blockIdx.x] != 0) != FAST) {
      if (MODE == kBwdFastTiles && blockIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      return;
    }
  }
  float a[NS], ra[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    a[k] = __ldg(p.A + static_cast<int64_t>(dc) * N + n0 + (k ^ perm));
    ra[k] = (a[k] != 0.0f) ? 1.0f / a[k] : 0.0f;
  }
  float nra[NS];  // -1/A: the packed coefficient (Abar - 1) / A = fma(Abar, 1/A, -1/A)
#pragma unroll
  for (int k = 0; k < NS; ++k) nra[k] = -ra[k];
  const float bias = p.bias ? __ldg(p.bias + dc) : 0.0f;
  const float Dd = p.D ? __ldg(p.D + dc) : 0.0f;

  IO rb[Cfg::BC_EPT], rc[Cfg::BC_EPT];
  if constexpr (PRE) {
    bwd_segment_pass<Cfg, FAST>(p, smem, seg, b, d0, chl, part, n0, perm, chv, row, rowbase,
                                rows, l_begin, j_begin, j_end, bias, a, ra);
  } else {
    // checkpoints of the state entering every block, in state order: the training
    // forward's, or those phase 1 writes below
    const float* ckr = p.ckpt_in ? p.ckpt_in : p.ckpt;
    // state entering the segment: h0, then each earlier segment i folded in as
    // h <- 2^(A sum_i) h + E_i (the recurrence is linear in h; 2^(A sum_i) is the
    // product of segment i's Abar factors)
    float h[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) h[k] = (chv && p.h0) ? p.h0[row * N + n0 + (k ^ perm)] : 0.0f;
    if (chv && !p.ckpt_in) {
#pragma unroll 1
      for (int i = 0; i < seg; ++i) {
        const float sum = p.seg_sum[i * rows + row];
        const float* E = p.seg_E + (i * rows + row) * N + n0;
#pragma unroll
        for (int k = 0; k < NS; ++k) h[k] = fmaf(ex2(a[k] * sum), h[k], E[k ^ perm]);
      }
    }

    const int nblk = j_end - j_begin;  // blocks of this segment
    // ---------------- phase 1: forward, checkpoint entering each block
    if (nblk > 0 && !p.ckpt_in) {
      bwd_stage<Cfg>(p, stage(0), rowbase, d0, l_begin, false);
      cp_async_commit();
      bwd_bc_fetch<Cfg>(p, b, l_begin, false, rb, rc);
      bwd_bc_park<Cfg>(bcbuf(0), rb, rc);
    }
    for (int jj = 0; jj < (p.ckpt_in ? 0 : nblk); ++jj) {
      const int j = j_begin + jj, l0 = j * kBwdPos, buf = jj & 1;
      cp_async_wait_all();
      __syncthreads();  // stage j and B of block j visible; block j-1 fully consumed
      const bool more = jj + 1 < nblk;
      if (more) {
        bwd_stage<Cfg>(p, stage(buf ^ 1), rowbase, d0, l0 + kBwdPos, false);
        cp_async_commit();
        bwd_bc_fetch<Cfg>(p, b, l0 + kBwdPos, false, rb, rc);
      }
      bwd_prologue<Cfg>(p, stage(buf), chl, part, bias, S, SG, false);
      if (chv) {
#pragma unroll
        for (int k = 0; k < NS; ++k)
          p.ckpt[(static_cast<int64_t>(j) * rows + row) * N + n0 + (k ^ perm)] = h[k];
      }
      __syncwarp();
      bwd_advance<Cfg, FAST>(p, stage(buf), bt(buf), S, chl, n0, l0, a, ra, h);
      if (more) bwd_bc_park<Cfg>(bcbuf(buf ^ 1), rb, rc);
    }

    // ---------------- phase 2: blocks in reverse
    float g[NS], an[NS], dA[NS], he[NS], hn[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      g[k] = (chv && p.dh_last) ? p.dh_last[row * N + n0 + (k ^ perm)] : 0.0f;
      an[k] = 1.0f;
      dA[k] = 0.0f;
      hn[k] = 0.0f;
    }
    // adjoint entering the segment from its end: dh_last, then each later segment i
    // folded in as g <- 2^(A sum_i) g + R_i (the adjoint is linear in g and passes
    // through segment i's Abar factors)
    if (chv) {
#pragma unroll 1
      for (int i = p.nseg - 1; i > seg; --i) {
        const float sum = p.seg_sum[i * rows + row];
        const float* R = p.seg_R + (i * rows + row) * N + n0;
#pragma unroll
        for (int k = 0; k < NS; ++k) g[k] = fmaf(ex2(a[k] * sum), g[k], R[k ^ perm]);
      }
    }
    float dD_acc = 0.0f, db_acc = 0.0f;
    __syncthreads();  // phase 1's last block consumed
    if (nblk > 0) {
      const int l0 = (j_end - 1) * kBwdPos;
      bwd_stage<Cfg>(p, stage(0), rowbase, d0, l0, true);
      cp_async_commit();
      bwd_bc_fetch<Cfg>(p, b, l0, true, rb, rc);
      bwd_bc_park<Cfg>(bcbuf(0), rb, rc);
      if (chv) {
#pragma unroll
        for (int k = 0; k < NS; ++k)
          hn[k] = ckr[(static_cast<int64_t>(j_end - 1) * rows + row) * N + n0 + (k ^ perm)];
      }
    }
    for (int it = 0; it < nblk; ++it) {
      const int j = j_end - 1 - it, l0 = j * kBwdPos, buf = it & 1;
      cp_async_wait_all();
      __syncthreads();  // stage of block j visible; the previous block fully consumed
#pragma unroll
      for (int k = 0; k < NS; ++k) he[k] = hn[k];
      const bool more = j > j_begin;
      if (more) {
        bwd_stage<Cfg>(p, stage(buf ^ 1), rowbase, d0, l0 - kBwdPos, true);
        cp_async_commit();
        bwd_bc_fetch<Cfg>(p, b, l0 - kBwdPos, true, rb, rc);
        if (chv) {
#pragma unroll
          for (int k = 0; k < NS; ++k)
            hn[k] = ckr[(static_cast<int64_t>(j - 1) * rows + row) * N + n0 + (k ^ perm)];
        }
      }
      bwd_prologue<Cfg>(p, stage(buf), chl, part, bias, S, SG, p.softplus != 0);
      __syncwarp();
      bwd_block<Cfg, FAST>(p, stage(buf), bt(buf), ct(buf), S, DY0, RED, WB, OUT, chl, part,
                           lane, warp, n0, l0, Dd, a, ra, nra, he, g, an, dA, dD_acc);
      __syncwarp();
      // per-position totals over the channel's four lanes: du (with the D skip) and
      // ddelta (through the softplus) for this lane's positions part*kBwdPpl ..
#pragma unroll
      for (int i = 0; i < kBwdPpl; ++i) {
        const int pp = part * kBwdPpl + i;
        if (l0 + pp < p.seqlen) {
          const float4 r0 = lds128f(RED + chl * Cfg::REDS + pp * 8);
          const float4 r1 = lds128f(RED + chl * Cfg::REDS + pp * 8 + 4);
          const float du = fmaf(Dd, DY0[chl * Cfg::SCS + pp], (r0.x + r0.y) + (r0.z + r0.w));
          float dx = (r1.x + r1.y) + (r1.z + r1.w);
          if (p.softplus) dx *= SG[chl * Cfg::SCS + pp];
          db_acc += dx;
          Io<IO>::store(reinterpret_cast<IO*>(OUT + chl * Cfg::ROWB) + pp, du);
          Io<IO>::store(reinterpret_cast<IO*>(OUT + Cfg::CHB + chl * Cfg::ROWB) + pp, dx);
        }
      }
      __syncthreads();  // WB and OUT complete
      // dB / dC partials of this CTA: sum the warps
      for (int v = tid; v < 2 * N * kBwdPos; v += Cfg::THREADS) {
        const int pp = v % kBwdPos, n = (v / kBwdPos) % N, t = v / (kBwdPos * N);
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < Cfg::WARPS; ++w) sum += WB[((w * 2 + t) * N + n) * Cfg::WBS + pp];
        const int l = l0 + pp;
        if (l < p.seqlen)
          p.part_bc[((static_cast<int64_t>(tile) * p.batch + b) * 2 + t) * N *
                        static_cast<int64_t>(p.seqlen) +
                    static_cast<int64_t>(n) * p.seqlen + l] = sum;
      }
      // du, ddelta, dz tiles
      {
        auto dst = [&](int t) -> IO* {
          return static_cast<IO*>(t == 0 ? p.du : t == 1 ? p.ddelta : p.dz);
        };
        const int ntens = Cfg::GATE ? 3 : 2;
        if constexpr (Cfg::VEC) {
          constexpr int CPR = Cfg::ROWB / 16, PPC = 16 / Cfg::ES;
          for (int c = tid; c < ntens * CH * CPR; c += Cfg::THREADS) {
            const int k = c % CPR, ch = (c / CPR) % CH, t = c / (CPR * CH);
            const int dd = d0 + ch, l = l0 + k * PPC;
            if (dd < p.dim && l < p.seqlen)
              *reinterpret_cast<uint4*>(dst(t) +
                                        (rowbase + dd) * static_cast<int64_t>(p.seqlen) + l) =
                  lds128(OUT + t * Cfg::CHB + ch * Cfg::ROWB + k * 16);
          }
        } else {
          for (int e = tid; e < ntens * CH * kBwdPos; e += Cfg::THREADS) {
            const int pp = e % kBwdPos, ch = (e / kBwdPos) % CH, t = e / (kBwdPos * CH);
            const int dd = d0 + ch, l = l0 + pp;
            if (dd < p.dim && l < p.seqlen)
              dst(t)[(rowbase + dd) * static_cast<int64_t>(p.seqlen) + l] =
                  reinterpret_cast<const IO*>(OUT + t * Cfg::CHB + ch * Cfg::ROWB)[pp];
          }
        }
      }
      if (more) bwd_bc_park<Cfg>(bcbuf(buf ^ 1), rb, rc);
    }

    // ---------------- per-channel results
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 1);
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 2);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 1);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 2);
    if (chv) {
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        p.part_a[(seg * rows + row) * N + n0 + (k ^ perm)] = dA[k];
        if (p.dh0 && seg == 0) p.dh0[row * N + n0 + (k ^ perm)] = an[k] * g[k];
      }
      if (part == 0) {
        p.part_dd[(seg * rows + row) * 2 + 0] = dD_acc;
        p.part_dd[(seg * rows + row) * 2 + 1] = db_acc;
      }
    }
  }
  if constexpr (MODE == kBwdFastTiles) {
    if (blockIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  }
}

// Per CTA of the gradient (segment, batch row, tile of 32 channels), whether the fast
// coefficients (Abar - 1) / A hold (bf16 io, ZOH): every |A| of its channels at least
// kFastPathMinAbsA, and every step of its positions with |q| = s |A| at least
// kBwdFastPathMinQ (s = dt log2 e; softplus is monotone, so the smallest raw step
// decides).  With Abar = ex2(q) the coefficient (Abar - 1) / A carries an error of
// about 2^-24 / |q ln 2| of itself (measured near the limit: below 0.5 %), so a tile
// whose steps vanish needs the series.
constexpr float kBwdFastPathMinQ = 1.52587890625e-05f;  // 2^-16

template <int N>
__global__ void __launch_bounds__(128) scan_bwd_classify_kernel(const BwdParams p, bool vec,
                                                                unsigned char* flags) {
  const int tid = threadIdx.x, chl = tid >> 2, part = tid & 3;
  const int64_t per_seg = p.batch * p.tiles;
  const int seg = static_cast<int>(blockIdx.x / per_seg);
  const int64_t b = (blockIdx.x % per_seg) / p.tiles;
  const int tile = static_cast<int>(blockIdx.x % p.tiles);
  const int d = tile * (128 / kBwdLpc) + chl;
  const int l_begin = seg * p.seg_len;
  const int l_end = (p.seqlen - l_begin < p.seg_len) ? p.seqlen : l_begin + p.seg_len;
  bool ok = true;
  if (d < p.dim) {
    float amin = fabsf(__ldg(p.A + static_cast<int64_t>(d) * N));
#pragma unroll
    for (int n = 1; n < N; ++n) amin = fminf(amin, fabsf(__ldg(p.A + static_cast<int64_t>(d) * N + n)));
    ok = amin >= kFastPathMinAbsA;
    if (ok) {
      const uint16_t* row = static_cast<const uint16_t*>(p.delta) +
                            (b * p.dim + d) * static_cast<int64_t>(p.seqlen);
      float xmin = 3.0e38f;
      if (vec) {
        // 16-byte rows: segment starts are multiples of 8 positions, and a vector
        // reaching past l_end stays inside the row (its length is a multiple of 8)
        for (int l = l_begin + part * 8; l < l_end; l += 32) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(row + l));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (l + 2 * k < l_end) xmin = fminf(xmin, bf16lo(ws[k]));
            if (l + 2 * k + 1 < l_end) xmin = fminf(xmin, bf16hi(ws[k]));
          }
        }
      } else {
        for (int l = l_begin + part; l < l_end; l += 4) xmin = fminf(xmin, bf16_to_f32(row[l]));
      }
      const float x2 = (xmin + (p.bias ? __ldg(p.bias + d) : 0.0f)) * kLog2e;
      const float s = p.softplus ? softplus_log2_accurate(x2) : x2;
      ok = s * amin >= kBwdFastPathMinQ;
    }
  }
  ok = __syncthreads_and(ok) != 0;
  if (tid == 0) flags[blockIdx.x] = ok ? 1 : 0;
}

// dB, dC [batch][N][seqlen] = sum over a batch row's CTAs of the partials, in
// CTA order.
template <typename IO>
__global__ void __launch_bounds__(256) scan_bwd_reduce_bc_kernel(const float* part, int tiles,
                                                                 int64_t batch, int N, int seqlen,
                                                                 IO* dB, IO* dC) {
  const int64_t per_tile = batch * 2 * N * static_cast<int64_t>(seqlen);
  const int64_t e = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (e >= per_tile) return;
  float sum = 0.0f;
  for (int t = 0; t < tiles; ++t) sum += part[t * per_tile + e];
  const int64_t ns = static_cast<int64_t>(N) * seqlen;
  const int64_t bt = e / ns, rem = e % ns;  // bt = b * 2 + (0: dB, 1: dC)
  IO* out = (bt & 1) ? dC : dB;
  Io<IO>::store(out + (bt >> 1) * ns + rem, sum);
}

// dA [dim][N], dD, bias gradient [dim] = sums over the batch rows, in row order
// (a template only so that every translation unit may include this header)
template <int kUnused = 0>
__global__ void __launch_bounds__(256) scan_bwd_reduce_param_kernel(
    const float* part_a, const float* part_dd, int64_t batch, int dim, int N, float* dA, float* dD,
    float* dbias) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const int64_t na = static_cast<int64_t>(dim) * N;
  if (i < na) {
    float s = 0.0f;
    for (int64_t b = 0; b < batch; ++b) s += part_a[b * na + i];
    dA[i] = s;
  } else if (i < na + dim) {
    const int64_t dd = i - na;
    float sd = 0.0f, sb = 0.0f;
    for (int64_t b = 0; b < batch; ++b) {
      sd += part_dd[(b * dim + dd) * 2];
      sb += part_dd[(b * dim + dd) * 2 + 1];
    }
    if (dD) dD[dd] = sd;
    if (dbias) dbias[dd] = sb;
  }
}

}  // namespace ssm
