// scan_channel.cuh -- selective-scan forward, "channel" kernel family.
//
// Mapping (B300, sm_103a): one lane owns one (batch, dim) channel and all of its
// N states, in registers, for the whole sequence.  The recurrence along L is
// then a plain sequential loop per lane: no cross-lane scan, no exchange, and
// N/2 independent packed (f32x2) state chains per position to hide latency.
// The (B, L, D, N) tensor never leaves registers (velog Mamba review, section
// 3.3 "Kernel Fusion": load the 3-D inputs to SRAM, discretise and recur there,
// write only the 3-D output).
//
// One CTA = 4 warps = 128 channels of one batch row.  L streams in chunks of
// RB bytes per row (16 or 32 bf16 positions, 8..32 fp32 positions):
//   * u, delta, z tiles [128 x chunk] and the B, C tiles [N x chunk] are loaded
//     by TMA (cp.async.bulk.tensor.3d, swizzle matching the row width, zero fill
//     past the tensor) into an S-stage ring; completion on mbarriers whose waits
//     are bounded in time and record a status bit on timeout;
//   * once per chunk the CTA re-lays B, C out as fp32 [position][state], so a
//     lane reads four states of one position with one 16-byte broadcast load;
//   * each lane reads 16-byte blocks of its row (8 bf16 / 4 fp32 positions),
//     runs the recurrence, adds D u, applies silu(z), rounds, and writes its y
//     block into a swizzled output tile that one thread stores by TMA.
//
// Discretisation (velog review, section 2 "Discretization"; "mamba 学习",
// section "MAMBA"): Abar = 2^(s A) with s = dt log2(e) (softplus evaluated in
// log2 units) and the ZOH input term (Abar - 1) / A * B u.  Fast path (bf16 io,
// every |A| >= 1/8 in the CTA):
//     w = B u / A,  h <- Abar (h + w) - w          (= Abar h + (Abar - 1) w)
// one ex2 and 6 fp32 lane-operations per state update.  Accurate path (fp32 io,
// or small / zero A): h <- Abar h + expm1(dt A) / A * B u with expm1 from its
// Taylor series near zero and the dt limit at A == 0.
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
  // raw pointers (used by the chunk kernel)
  const void* u;
  const void* delta;
  const void* z;
  const void* B;
  const void* C;
  void* y;
};

// |A| below this (or A == 0) sends a bf16 CTA to the accurate path: the fast
// path forms (Abar - 1) w as Abar (h + w) - w, whose absolute error grows like
// 2^-22 |B u / A|.
constexpr float kFastPathMinAbsA = 0.125f;

template <typename IO, int N_, bool GATE_, int S_, int RB_>
struct ChanCfg {
  static constexpr int N = N_;
  static constexpr bool GATE = GATE_;
  static constexpr int S = S_;              // pipeline stages
  static constexpr int RB = RB_;            // bytes of one row of a chunk (32, 64 or 128)
  static_assert(RB == 32 || RB == 64 || RB == 128, "row width must be a TMA swizzle span");
  static_assert(N % 4 == 0, "dstate must be a multiple of 4");
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int DT = THREADS;        // channels per CTA (one per lane)
  static constexpr int ESZ = Io<IO>::kBytes;
  static constexpr int TB = 16 / ESZ;       // positions per 16-byte block
  static constexpr int LC = RB / ESZ;       // positions per chunk
  static constexpr int NBLK = RB / 16;      // 16-byte blocks per row
  static constexpr int NARR = GATE ? 3 : 2; // u, delta (, z)
  static constexpr int pad1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int TILE = pad1k(DT * RB);      // one [DT x LC] swizzled tile
  static constexpr int BCT = pad1k(N * RB);        // one [N x LC] swizzled tile
  static constexpr int STAGE = NARR * TILE + 2 * BCT;
  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_Y = OFF_STAGES + S * STAGE;          // 2 output tiles
  static constexpr int BCF = LC * N * 4;                        // fp32 [LC][N]
  static constexpr int OFF_BCF = OFF_Y + 2 * TILE;              // [2 buf][B, C]
  static constexpr int OFF_BAR = OFF_BCF + 2 * 2 * BCF;
  static constexpr int SMEM = OFF_BAR + S * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;                // for base alignment
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
  static constexpr uint32_t TX_BYTES = NARR * DT * RB + 2 * N * RB;
};

struct ChanMaps {
  CUtensorMap u, delta, z, y, B, C;
};

// Byte offset of 16-byte granule c of row r in a tile of RB-byte rows written by
// TMA with the swizzle of span RB (tile base 1024-byte aligned): the granule
// index is XOR-ed with address bits 7 and up.
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * RB + ((c ^ (((r * RB) >> 7) & (RB / 16 - 1))) << 4);
}

template <typename IO, int TB>
__device__ __forceinline__ void unpack16(const uint4 w, float* out) {
  if constexpr (sizeof(IO) == 2) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = bf16lo(ws[k]);
      out[2 * k + 1] = bf16hi(ws[k]);
    }
  } else {
    out[0] = __uint_as_float(w.x);
    out[1] = __uint_as_float(w.y);
    out[2] = __uint_as_float(w.z);
    out[3] = __uint_as_float(w.w);
  }
}

template <typename IO, int TB>
__device__ __forceinline__ uint4 pack16(const float* v) {
  if constexpr (sizeof(IO) == 2) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                      pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  } else {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
  }
}

// ---------------------------------------------------------------------------
// one chunk of positions for one lane (its channel's row `row` of the tiles)
// ---------------------------------------------------------------------------
template <typename Cfg, typename IO, bool ACC, bool TAIL>
__device__ __forceinline__ void chan_chunk(const uint8_t* stage, uint8_t* ytile, const float* bcfB,
                                           const float* bcfC, int row, int l0, int seqlen,
                                           const float* Areg, const float* nIA, float Dd,
                                           float bias2, int softplus, float* h) {
  constexpr int N = Cfg::N, TB = Cfg::TB, RB = Cfg::RB;
  const uint8_t* tu = stage;
  const uint8_t* td = stage + Cfg::TILE;
  const uint8_t* tz = stage + 2 * Cfg::TILE;

#pragma unroll 1
  for (int blk = 0; blk < Cfg::NBLK; ++blk) {
    const uint32_t off = swz<RB>(row, blk);
    float uj[TB], sj[TB];
    unpack16<IO, TB>(lds128(tu + off), uj);
    unpack16<IO, TB>(lds128(td + off), sj);
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const float x2 = fmaf(sj[j], kLog2e, bias2);
      float s = softplus ? (ACC ? softplus_log2_accurate(x2) : softplus_log2_fast(x2)) : x2;
      if constexpr (TAIL) s = (l0 + blk * TB + j < seqlen) ? s : 0.0f;  // past the end: Abar = 1
      sj[j] = s;
    }
    float yo[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int lc = blk * TB + j;  // position within the chunk
      const float* Bp = bcfB + lc * N;
      const float* Cp = bcfC + lc * N;
      f2 acc = mk2(0.0f, 0.0f);
#pragma unroll
      for (int m = 0; m < N; m += 4) {
        const float4 Bv = lds128f(Bp + m);
        const float4 Cv = lds128f(Cp + m);
        const float bv[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
        const float cv[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
#pragma unroll
        for (int pp = 0; pp < 4; pp += 2) {
          const int i = m + pp;
          if constexpr (!ACC) {
            const f2 q = mul2(mk2(sj[j], sj[j]), mk2(Areg[i], Areg[i + 1]));
            const f2 a = mk2(ex2(q.x), ex2(q.y));
            const f2 X = mul2(mk2(bv[pp], bv[pp + 1]), mk2(uj[j], uj[j]));
            const f2 nw = mul2(X, mk2(nIA[i], nIA[i + 1]));       // -w = -B u / A
            const f2 t = sub2(mk2(h[i], h[i + 1]), nw);           // h + w
            const f2 hn = fma2(a, t, nw);                         // Abar (h + w) - w
            h[i] = hn.x;
            h[i + 1] = hn.y;
          } else {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float A0 = Areg[i + e];
              const float q = sj[j] * A0;
              const float ahw = ex2(q);
              const float em1 = exp2m1_accurate(q, ahw);
              const float a = (fabsf(q) < 0.36f) ? 1.0f + em1 : ahw;
              // (Abar - 1) / A, or dt at A == 0
              const float coef = (A0 == 0.0f) ? sj[j] * kLn2 : em1 * -nIA[i + e];
              h[i + e] = fmaf(a, h[i + e], coef * (bv[pp + e] * uj[j]));
            }
          }
          acc = fma2(mk2(cv[pp], cv[pp + 1]), mk2(h[i], h[i + 1]), acc);
        }
      }
      yo[j] = fmaf(Dd, uj[j], acc.x + acc.y);
    }
    if constexpr (Cfg::GATE) {
      float zj[TB];
      unpack16<IO, TB>(lds128(tz + off), zj);
#pragma unroll
      for (int j = 0; j < TB; ++j) yo[j] *= (ACC ? silu_accurate(zj[j]) : silu_fast(zj[j]));
    }
    *reinterpret_cast<uint4*>(ytile + off) = pack16<IO, TB>(yo);
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename IO, typename Cfg>
__global__ void __launch_bounds__(Cfg::THREADS)
    scan_channel_kernel(const __grid_constant__ ChanMaps maps, const ScanParams p) {
  constexpr int N = Cfg::N, S = Cfg::S, LC = Cfg::LC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

  const int tid = threadIdx.x;
  const int b = blockIdx.x / p.dtiles;
  const int d0 = (blockIdx.x % p.dtiles) * Cfg::DT;
  const int row = tid;
  const int d = d0 + row;
  const bool valid = d < p.dim;
  const int nchunks = (p.seqlen + LC - 1) / LC;

  // per-lane parameters and state
  float Areg[N], nIA[N], h[N];
  bool small_a = false;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float a = valid ? __ldg(p.A + static_cast<int64_t>(d) * N + i) : -1.0f;
    Areg[i] = a;
    nIA[i] = (a == 0.0f) ? 0.0f : -1.0f / a;
    small_a |= !(fabsf(a) >= kFastPathMinAbsA);
    h[i] = (valid && p.h0) ? __ldg(p.h0 + (static_cast<int64_t>(b) * p.dim + d) * N + i) : 0.0f;
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

  int issued = (S < nchunks) ? S : nchunks;  // chunks whose loads were issued (thread 0)
  if (tid == 0)
    for (int k = 0; k < issued; ++k) issue_loads(k);

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
      const uint8_t* raw = st + Cfg::NARR * Cfg::TILE;
#pragma unroll 1
      for (int piece = tid; piece < 2 * N * Cfg::NBLK; piece += Cfg::THREADS) {
        const int arr = piece / (N * Cfg::NBLK);
        const int rem = piece % (N * Cfg::NBLK);
        const int n = rem % N, kb = rem / N;
        float v[Cfg::TB];
        unpack16<IO, Cfg::TB>(lds128(raw + arr * Cfg::BCT + swz<Cfg::RB>(n, kb)), v);
        float* dst = bf + arr * (Cfg::BCF / 4) + (kb * Cfg::TB) * N + n;
#pragma unroll
        for (int e = 0; e < Cfg::TB; ++e) dst[e * N] = v[e];
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
    const bool tail = (k + 1) * LC > p.seqlen;
    if constexpr (sizeof(IO) == 2) {
      if (!accurate) {
        if (!tail)
          chan_chunk<Cfg, IO, false, false>(st, ytile, bcfB, bcfC, row, k * LC, p.seqlen, Areg,
                                            nIA, Dd, bias2, p.softplus, h);
        else
          chan_chunk<Cfg, IO, false, true>(st, ytile, bcfB, bcfC, row, k * LC, p.seqlen, Areg,
                                           nIA, Dd, bias2, p.softplus, h);
      } else {
        chan_chunk<Cfg, IO, true, true>(st, ytile, bcfB, bcfC, row, k * LC, p.seqlen, Areg, nIA,
                                        Dd, bias2, p.softplus, h);
      }
    } else {
      chan_chunk<Cfg, IO, true, true>(st, ytile, bcfB, bcfC, row, k * LC, p.seqlen, Areg, nIA,
                                      Dd, bias2, p.softplus, h);
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
    for (int i = 0; i < N; ++i)
      p.h_last[(static_cast<int64_t>(b) * p.dim + d) * N + i] = h[i];
  }
}

}  // namespace ssm
