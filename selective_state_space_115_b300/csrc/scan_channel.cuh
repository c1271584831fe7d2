// scan_channel.cuh -- selective-scan forward, "channel" kernel family.
//
// Mapping (B300, sm_103a): every (batch, dim) channel's recurrence runs
// sequentially along L inside G lanes of one warp; lane g of a channel owns
// NS = N / G of its states in registers for the whole sequence, so no
// cross-lane scan is needed and the (B, L, D, N) state never leaves registers
// (velog Mamba review, section 3.3 "Kernel Fusion": load the 3-D inputs to
// SRAM, discretise and recur there, write only the 3-D output).
//
// One CTA = 4 warps = DT channels of one batch row, L streamed in chunks of one
// 128-byte row per channel (64 bf16 or 32 fp32 positions):
//   * u, delta, z tiles [DT x chunk] and the B, C tiles [N x chunk] are loaded
//     by TMA (cp.async.bulk.tensor, 128-byte swizzle) into an S-stage ring,
//     completion tracked by mbarriers (bounded waits);
//   * B, C are re-laid out once per chunk as fp32 [position][state], so a lane
//     reads its states of one position with one 16-byte broadcast load;
//   * per 16-byte block of positions, lane g of a channel computes softplus for
//     its share of positions and the lanes swap (dt, u) through shared memory;
//   * the C-contraction partials of the G lanes are summed through shared
//     memory; the lane that owns a position adds D u, applies silu(z), rounds,
//     and writes y into a swizzled output tile that one thread stores by TMA.
//
// Discretisation (velog review, section 2 "Discretization"; "mamba 学习",
// section "MAMBA"):  Abar = 2^(s A) with s = dt log2(e) (softplus evaluated in
// log2 units), and the ZOH input term (Abar - 1) / A * B u.  Fast path (bf16 io):
//     w = B u / A,  h <- Abar (h + w) - w          (= Abar h + (Abar - 1) w)
// 6 fp32 operations and one ex2 per state update.  Accurate path (fp32 io, or
// any |A| < 1/8 in the CTA, or A == 0):  h <- Abar h + expm1-accurate(s A)/A B u
// with the dt limit at A == 0.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

struct ScanParams {
  int batch, dim, seqlen;
  int dtiles;               // ceil(dim / DT)
  int softplus;
  const float* A;           // [dim, N]
  const float* D;           // [dim] or null
  const float* bias;        // [dim] or null
  const float* h0;          // [batch, dim, N] or null
  float* h_last;            // [batch, dim, N] or null
  DeviceStatus* status;
  // raw pointers (chunk kernel, and the TMA kernel's fallback-free paths)
  const void* u;
  const void* delta;
  const void* z;
  const void* B;
  const void* C;
  void* y;
};

// |A| below this (or A == 0) sends a bf16 CTA to the accurate path: the fast
// path computes (Abar - 1) w as Abar (h + w) - w, whose absolute error grows
// like 2^-22 |B u / A|.
constexpr float kFastPathMinAbsA = 0.125f;

template <typename IO, int N_, int G_, bool GATE_, int S_>
struct ChanCfg {
  static constexpr int N = N_;
  static constexpr int G = G_;
  static constexpr int NS = N / G;          // states per lane
  static constexpr bool GATE = GATE_;
  static constexpr int S = S_;              // pipeline stages
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int CPW = 32 / G;        // channels per warp
  static constexpr int DT = WARPS * CPW;    // channels per CTA
  static constexpr int ESZ = Io<IO>::kBytes;
  static constexpr int TB = 16 / ESZ;       // positions per 16-byte block
  static constexpr int LC = 128 / ESZ;      // positions per chunk
  static constexpr int NBLK = 8;            // 16-byte blocks per chunk row
  static constexpr int OWN = TB / G;        // positions a lane finalises per block
  static_assert(N % G == 0 && NS % 4 == 0, "states per lane must be a multiple of 4");
  static_assert(TB % G == 0, "a block must split evenly over the lanes of a channel");
  static constexpr int NARR = GATE ? 3 : 2;  // u, delta (, z)
  static constexpr int pad1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int TILE = pad1k(DT * 128);     // one [DT x LC] swizzled tile
  static constexpr int BCT = pad1k(N * 128);       // one [N x LC] swizzled tile
  static constexpr int STAGE = NARR * TILE + 2 * BCT;
  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_Y = OFF_STAGES + S * STAGE;            // 2 output tiles
  static constexpr int BCF = LC * N * 4;                          // fp32 [LC][N]
  static constexpr int OFF_BCF = OFF_Y + 2 * TILE;                // [2 buf][B, C]
  // lane exchange buffers (only when a channel spans several lanes)
  static constexpr int SU_ROW = TB * 16 + 16;                     // (dt, dt, u, u) + pad
  static constexpr int SU_WARP = (G > 1) ? CPW * SU_ROW : 0;
  static constexpr int OFF_SU = OFF_BCF + 2 * 2 * BCF;            // [warp][2 buf]
  static constexpr int RED_ROW = 36 * 4;                          // 32 lanes + pad
  static constexpr int RED_WARP = (G > 1) ? TB * RED_ROW : 0;
  static constexpr int OFF_RED = OFF_SU + WARPS * 2 * SU_WARP;    // [warp][2 buf]
  static constexpr int OFF_BAR = (OFF_RED + WARPS * 2 * RED_WARP + 15) / 16 * 16;
  static constexpr int SMEM = OFF_BAR + S * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;                  // for base alignment
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
  static constexpr uint32_t TX_BYTES = NARR * DT * 128 + 2 * N * 128;
};

struct ChanMaps {
  CUtensorMap u, delta, z, y, B, C;
};

// ---------------------------------------------------------------------------
// one chunk of positions for one lane
// ---------------------------------------------------------------------------
// raw io value(s) of this lane's own positions in a 16-byte block, as fp32
template <typename IO, int OWN>
__device__ __forceinline__ void load_own(const uint8_t* p, float* out) {
  if constexpr (sizeof(IO) == 2) {
    if constexpr (OWN == 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      out[0] = bf16lo(w);
      out[1] = bf16hi(w);
    } else if constexpr (OWN == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      out[0] = bf16lo(w.x); out[1] = bf16hi(w.x); out[2] = bf16lo(w.y); out[3] = bf16hi(w.y);
    } else {
      const uint4 w = lds128(p);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) { out[2 * k] = bf16lo(ws[k]); out[2 * k + 1] = bf16hi(ws[k]); }
    }
  } else {
    if constexpr (OWN == 1) {
      out[0] = *reinterpret_cast<const float*>(p);
    } else if constexpr (OWN == 2) {
      const float2 w = *reinterpret_cast<const float2*>(p);
      out[0] = w.x; out[1] = w.y;
    } else {
      const float4 w = lds128f(p);
      out[0] = w.x; out[1] = w.y; out[2] = w.z; out[3] = w.w;
    }
  }
}

template <typename Cfg, typename IO, bool ACC>
__device__ __forceinline__ void chan_chunk(const uint8_t* stage, uint8_t* ytile, const float* bcfB,
                                           const float* bcfC, uint8_t* su_base, uint8_t* red_base,
                                           int warp, int lane, int c, int g, int l0, int seqlen,
                                           const float* Areg, const float* nIA, const float* IA,
                                           const float* isZ, float Dd, float bias2, int softplus,
                                           float* h) {
  constexpr int NS = Cfg::NS, G = Cfg::G, TB = Cfg::TB, OWN = Cfg::OWN, N = Cfg::N;
  constexpr int ESZ = Cfg::ESZ;
  const int row = warp * Cfg::CPW + c;
  const uint8_t* tu = stage;
  const uint8_t* td = stage + Cfg::TILE;
  const uint8_t* tz = stage + 2 * Cfg::TILE;
  const int own0 = (G == 1) ? 0 : g * OWN;  // first position of the block this lane finalises

#pragma unroll 1
  for (int blk = 0; blk < Cfg::NBLK; ++blk) {
    const uint32_t off = swz128(row, blk) + own0 * ESZ;
    const int lb = l0 + blk * TB;  // first position of this block
    // ---- dt (log2 units) and u of this lane's own positions
    float uo[OWN], dto[OWN];
    load_own<IO, OWN>(tu + off, uo);
    load_own<IO, OWN>(td + off, dto);
#pragma unroll
    for (int k = 0; k < OWN; ++k) {
      const float x2 = fmaf(dto[k], kLog2e, bias2);
      const float s = softplus ? (ACC ? softplus_log2_accurate(x2) : softplus_log2_fast(x2)) : x2;
      dto[k] = (lb + own0 + k < seqlen) ? s : 0.0f;  // past the end: Abar = 1, no input
    }
    // ---- every position's (dt, dt, u, u) for the recurrence
    float4 su[TB];
    if constexpr (G == 1) {
#pragma unroll
      for (int j = 0; j < TB; ++j) su[j] = make_float4(dto[j], dto[j], uo[j], uo[j]);
    } else {
      uint8_t* sub = su_base + (blk & 1) * Cfg::SU_WARP + c * Cfg::SU_ROW;
#pragma unroll
      for (int k = 0; k < OWN; ++k)
        *reinterpret_cast<float4*>(sub + (own0 + k) * 16) = make_float4(dto[k], dto[k], uo[k], uo[k]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < TB; ++j) su[j] = lds128f(sub + j * 16);
    }
    // ---- recurrence over the block: NS states, TB positions
    float yp[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int lc = blk * TB + j;  // position within chunk
      const float* Bp = bcfB + lc * N + g * NS;
      const float* Cp = bcfC + lc * N + g * NS;
      const f2 ss = mk2(su[j].x, su[j].y);
      const f2 uu = mk2(su[j].z, su[j].w);
      float acc = 0.0f;
#pragma unroll
      for (int m = 0; m < NS; m += 4) {
        const float4 Bv = lds128f(Bp + m);
        const float4 Cv = lds128f(Cp + m);
        const float bvals[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
        const float cvals[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
#pragma unroll
        for (int pp = 0; pp < 4; pp += 2) {
          const int i = m + pp;
          if constexpr (!ACC) {
            const f2 q = mul2(ss, mk2(Areg[i], Areg[i + 1]));
            const f2 a = mk2(ex2(q.x), ex2(q.y));
            const f2 X = mul2(mk2(bvals[pp], bvals[pp + 1]), uu);
            const f2 nw = mul2(X, mk2(nIA[i], nIA[i + 1]));        // -w = -B u / A
            const f2 t = sub2(mk2(h[i], h[i + 1]), nw);            // h + w
            const f2 hn = fma2(a, t, nw);                          // Abar (h + w) - w
            h[i] = hn.x;
            h[i + 1] = hn.y;
          } else {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float q = su[j].x * Areg[i + e];
              const float ahw = ex2(q);
              const float em1 = exp2m1_accurate(q, ahw);
              const float a = (fabsf(q) < 0.36f) ? 1.0f + em1 : ahw;
              float coef = em1 * IA[i + e];
              coef = fmaf(isZ[i + e], su[j].x * kLn2, coef);        // dt at A == 0
              h[i + e] = fmaf(a, h[i + e], coef * (bvals[pp + e] * su[j].z));
            }
          }
          acc = fmaf(cvals[pp], h[i], acc);
          acc = fmaf(cvals[pp + 1], h[i + 1], acc);
        }
      }
      yp[j] = acc;
    }
    // ---- sum the G partial contractions; finalise this lane's positions
    float ysum[OWN];
    if constexpr (G == 1) {
#pragma unroll
      for (int j = 0; j < TB; ++j) ysum[j] = yp[j];
    } else {
      uint8_t* red = red_base + (blk & 1) * Cfg::RED_WARP;
#pragma unroll
      for (int j = 0; j < TB; ++j) *reinterpret_cast<float*>(red + j * Cfg::RED_ROW + lane * 4) = yp[j];
      __syncwarp();
#pragma unroll
      for (int k = 0; k < OWN; ++k) {
        const uint8_t* src = red + (own0 + k) * Cfg::RED_ROW + c * G * 4;
        float sacc;
        if constexpr (G == 4) {
          const float4 v = lds128f(src);
          sacc = (v.x + v.y) + (v.z + v.w);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          sacc = v.x + v.y;
        }
        ysum[k] = sacc;
      }
    }
    float yo[OWN];
    float zo[OWN];
    if constexpr (Cfg::GATE) load_own<IO, OWN>(tz + off, zo);
#pragma unroll
    for (int k = 0; k < OWN; ++k) {
      float v = fmaf(Dd, uo[k], ysum[k]);
      if constexpr (Cfg::GATE) v *= (ACC ? silu_accurate(zo[k]) : silu_fast(zo[k]));
      yo[k] = v;
    }
    uint8_t* ydst = ytile + off;
    if constexpr (sizeof(IO) == 2) {
      if constexpr (OWN == 8) {
        *reinterpret_cast<uint4*>(ydst) =
            make_uint4(pack_bf16x2(yo[0], yo[1]), pack_bf16x2(yo[2], yo[3]),
                       pack_bf16x2(yo[4], yo[5]), pack_bf16x2(yo[6], yo[7]));
      } else if constexpr (OWN == 4) {
        *reinterpret_cast<uint2*>(ydst) =
            make_uint2(pack_bf16x2(yo[0], yo[1]), pack_bf16x2(yo[2], yo[3]));
      } else {
        *reinterpret_cast<uint32_t*>(ydst) = pack_bf16x2(yo[0], yo[1]);
      }
    } else {
      if constexpr (OWN == 4) {
        *reinterpret_cast<float4*>(ydst) = make_float4(yo[0], yo[1], yo[2], yo[3]);
      } else if constexpr (OWN == 2) {
        *reinterpret_cast<float2*>(ydst) = make_float2(yo[0], yo[1]);
      } else {
        *reinterpret_cast<float*>(ydst) = yo[0];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename IO, typename Cfg>
__global__ void __launch_bounds__(Cfg::THREADS)
    scan_channel_kernel(const __grid_constant__ ChanMaps maps, const ScanParams p) {
  constexpr int N = Cfg::N, NS = Cfg::NS, G = Cfg::G, S = Cfg::S, LC = Cfg::LC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = lane / G, g = lane % G;
  const int b = blockIdx.x / p.dtiles;
  const int d0 = (blockIdx.x % p.dtiles) * Cfg::DT;
  const int row = warp * Cfg::CPW + c;
  const int d = d0 + row;
  const bool valid = d < p.dim;
  const int nchunks = (p.seqlen + LC - 1) / LC;

  // per-lane parameters
  float Areg[NS], nIA[NS], IA[NS], isZ[NS], h[NS];
  bool small_a = false;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float a = valid ? __ldg(p.A + static_cast<int64_t>(d) * N + g * NS + i) : -1.0f;
    Areg[i] = a;
    const bool z0 = (a == 0.0f);
    IA[i] = z0 ? 0.0f : 1.0f / a;
    nIA[i] = -IA[i];
    isZ[i] = z0 ? 1.0f : 0.0f;
    small_a |= !(fabsf(a) >= kFastPathMinAbsA);
    h[i] = (valid && p.h0) ? __ldg(p.h0 + (static_cast<int64_t>(b) * p.dim + d) * N + g * NS + i)
                           : 0.0f;
  }
  const float Dd = (valid && p.D) ? __ldg(p.D + d) : 0.0f;
  const float bias2 = (valid && p.bias) ? __ldg(p.bias + d) * kLog2e : 0.0f;
  const bool accurate = (sizeof(IO) == 4) ? true : (__syncthreads_or(small_a) != 0);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.delta);
    prefetch_tmap(&maps.B);
    prefetch_tmap(&maps.C);
    prefetch_tmap(&maps.y);
    if (Cfg::GATE) prefetch_tmap(&maps.z);
  }
  __syncthreads();

  auto issue_loads = [&](int k) {
    uint8_t* st = smem + Cfg::OFF_STAGES + (k % S) * Cfg::STAGE;
    uint64_t* bar = &full[k % S];
    mbar_arrive_expect_tx(bar, Cfg::TX_BYTES);
    const int l = k * LC;
    tma_load_3d(st, &maps.u, bar, l, d0, b);
    tma_load_3d(st + Cfg::TILE, &maps.delta, bar, l, d0, b);
    if (Cfg::GATE) tma_load_3d(st + 2 * Cfg::TILE, &maps.z, bar, l, d0, b);
    tma_load_3d(st + Cfg::NARR * Cfg::TILE, &maps.B, bar, l, 0, b);
    tma_load_3d(st + Cfg::NARR * Cfg::TILE + Cfg::BCT, &maps.C, bar, l, 0, b);
  };

  if (tid == 0) {
    for (int k = 0; k < S && k < nchunks; ++k) issue_loads(k);
  }

  uint8_t* su_base = smem + Cfg::OFF_SU + warp * 2 * Cfg::SU_WARP;
  uint8_t* red_base = smem + Cfg::OFF_RED + warp * 2 * Cfg::RED_WARP;
  int issued = (S < nchunks) ? S : nchunks;  // chunks whose loads were issued (thread 0's view)
  int k = 0;
  bool ok = true;

  for (; k < nchunks; ++k) {
    const int s = k % S;
    const uint8_t* st = smem + Cfg::OFF_STAGES + s * Cfg::STAGE;
    const bool arrived = mbar_wait_bounded(&full[s], (k / S) & 1);
    if (!arrived) record_timeout(p.status, 1u);
    // B, C of this chunk: swizzled [N][LC] io -> fp32 [LC][N]
    {
      float* bf = reinterpret_cast<float*>(smem + Cfg::OFF_BCF + (k & 1) * 2 * Cfg::BCF);
      const uint8_t* rawB = st + Cfg::NARR * Cfg::TILE;
#pragma unroll 1
      for (int piece = tid; piece < 2 * N * 8; piece += Cfg::THREADS) {
        const int arr = piece / (N * 8);
        const int rem = piece % (N * 8);
        const int n = rem % N, kb = rem / N;
        const uint4 v = lds128(rawB + arr * Cfg::BCT + swz128(n, kb));
        float* dst = bf + arr * (Cfg::BCF / 4);
        if constexpr (sizeof(IO) == 2) {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dst[(kb * 8 + 2 * e) * N + n] = bf16lo(w[e]);
            dst[(kb * 8 + 2 * e + 1) * N + n] = bf16hi(w[e]);
          }
        } else {
          dst[(kb * 4 + 0) * N + n] = __uint_as_float(v.x);
          dst[(kb * 4 + 1) * N + n] = __uint_as_float(v.y);
          dst[(kb * 4 + 2) * N + n] = __uint_as_float(v.z);
          dst[(kb * 4 + 3) * N + n] = __uint_as_float(v.w);
        }
      }
    }
    if (tid == 0 && k >= 2) tma_store_wait_read<0>();  // store of chunk k-2 has read its tile
    if (__syncthreads_or(!arrived)) {
      ok = false;
      break;
    }
    if (tid == 0 && k >= 1) {
      tma_store_3d(&maps.y, smem + Cfg::OFF_Y + ((k - 1) & 1) * Cfg::TILE, (k - 1) * LC, d0, b);
      tma_store_commit();
      if (k - 1 + S < nchunks) {
        fence_proxy_async_smem();
        issue_loads(k - 1 + S);  // stage of chunk k-1 is free: every thread passed the barrier
        ++issued;
      }
    }
    const float* bcfB =
        reinterpret_cast<const float*>(smem + Cfg::OFF_BCF + (k & 1) * 2 * Cfg::BCF);
    const float* bcfC = bcfB + Cfg::BCF / 4;
    uint8_t* ytile = smem + Cfg::OFF_Y + (k & 1) * Cfg::TILE;
    if constexpr (sizeof(IO) == 2) {
      if (!accurate)
        chan_chunk<Cfg, IO, false>(st, ytile, bcfB, bcfC, su_base, red_base, warp, lane, c, g,
                                   k * LC, p.seqlen, Areg, nIA, IA, isZ, Dd, bias2, p.softplus, h);
      else
        chan_chunk<Cfg, IO, true>(st, ytile, bcfB, bcfC, su_base, red_base, warp, lane, c, g,
                                  k * LC, p.seqlen, Areg, nIA, IA, isZ, Dd, bias2, p.softplus, h);
    } else {
      chan_chunk<Cfg, IO, true>(st, ytile, bcfB, bcfC, su_base, red_base, warp, lane, c, g, k * LC,
                                p.seqlen, Areg, nIA, IA, isZ, Dd, bias2, p.softplus, h);
    }
    fence_proxy_async_smem();  // y tile writes -> visible to the TMA store
  }
  __syncthreads();
  if (tid == 0) {
    if (ok && nchunks > 0) {
      tma_store_3d(&maps.y, smem + Cfg::OFF_Y + ((nchunks - 1) & 1) * Cfg::TILE,
                   (nchunks - 1) * LC, d0, b);
      tma_store_commit();
    }
    tma_store_wait_all<0>();
    if (!ok) {
      // a wait gave up at chunk k: before the CTA exits, wait (bounded) for every
      // load that may still be in flight into the ring (chunks k .. issued-1)
      for (int kk = k; kk < issued; ++kk) (void)mbar_wait_bounded(&full[kk % S], (kk / S) & 1);
    }
  }
  if (ok && valid && p.h_last) {
#pragma unroll
    for (int i = 0; i < NS; ++i)
      p.h_last[(static_cast<int64_t>(b) * p.dim + d) * N + g * NS + i] = h[i];
  }
}

}  // namespace ssm
