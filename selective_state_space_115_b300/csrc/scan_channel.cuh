// scan_channel.cuh -- selective-scan forward, "channel" kernel family.
//
// Mapping (B300, sm_103a): LPC lanes (1, 2 or 4, adjacent in the warp) own one
// (batch, dim) channel; each of them holds NS = N / LPC of its states in
// registers for the whole sequence.  The recurrence along L is a plain
// sequential loop per lane -- no cross-lane scan -- with NS/2 independent packed
// (f32x2) state chains per position to hide latency.  The (B, L, D, N) tensor
// never leaves registers (velog Mamba review, section 3.3 "Kernel Fusion": load
// the 3-D inputs to SRAM, discretise and recur there, write only the 3-D output).
//
// Splitting a channel over 2 or 4 lanes gives 2x / 4x more, shorter warps: more
// latency hiding per SM sub-partition and finer load balance over the 148 SMs.
// The per-position work (softplus, D skip, gate, rounding, store) is split over
// the LPC lanes too -- each takes TB/LPC positions of every 16-byte block -- and
// two short xor-shuffle exchanges join them: an all-gather of the step sizes
// before the recurrence and a reduce-scatter of the partial contractions after.
//
// One CTA = 4 warps = 128 / LPC channels of one batch row.  L streams in chunks
// of RB bytes per row:
//   * u, delta, z tiles [DT x chunk] and the B, C tiles [N x chunk] are loaded
//     by TMA (cp.async.bulk.tensor.3d, swizzle matching the row width, zero fill
//     past the tensor) into an S-stage ring; completion on mbarriers whose waits
//     are bounded in time and record a status bit on timeout;
//   * once per chunk the CTA re-lays B, C out as fp32 [position][state], so a
//     lane reads four states of one position with one 16-byte broadcast load;
//   * each lane stores its finished positions of y straight to global memory (16
//     bytes per block of positions at one lane per channel): no output tile, so
//     the CTA's shared memory holds the input ring alone.
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
  // L split across CTAs (segmented two-pass scan); nseg = 1, seg_len = seqlen otherwise
  int nseg;                 // segments of the sequence
  int seg_len;              // positions per segment (a multiple of the chunk)
  float* seg_state;         // [nseg][batch * dim][N]: end state of each segment from h = 0
  float* seg_sum;           // [nseg][batch * dim]: sum of dt * log2(e) over each segment
  // training forward: the state entering every block of kCkptPos positions,
  // [ceil(seqlen / kCkptPos)][batch * dim][N] fp32 (null: not written)
  float* ckpt;
};

// positions per state checkpoint of the training forward (the gradient's block)
constexpr int kCkptPos = 8;

// Kernel modes of the channel kernel:
//   kModeFull    one pass over the whole sequence (nseg = 1)
//   kModeStates  pass 1 of the segmented scan: each CTA runs its segment from a zero
//                state, reads u, delta, B only, and writes the segment's end state and
//                step-size sum (no output)
//   kModeCarry   pass 2: each CTA rebuilds the state entering its segment from h0 and
//                the earlier segments' (end state, step-size sum), then runs the
//                segment with outputs
constexpr int kModeFull = 0, kModeStates = 1, kModeCarry = 2;


template <typename IO, int N_, bool GATE_, int LPC_, int S_, int RB_, bool EULER_ = false>
struct ChanCfg {
  static constexpr int N = N_;
  static constexpr bool GATE = GATE_;
  static constexpr bool EULER = EULER_;     // input term dt * B instead of the ZOH form
  static constexpr int LPC = LPC_;          // lanes per channel
  static constexpr int NS = N / LPC;        // states per lane
  static constexpr int S = S_;              // pipeline stages
  static constexpr int RB = RB_;            // bytes of one row of a chunk (32, 64 or 128)
  static_assert(RB == 32 || RB == 64 || RB == 128, "row width must be a TMA swizzle span");
  static_assert(LPC == 1 || LPC == 2 || LPC == 4, "1, 2 or 4 lanes per channel");
  static_assert(NS % 4 == 0, "each lane holds a multiple of 4 states");
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int DT = THREADS / LPC;  // channels per CTA
  static constexpr int ESZ = Io<IO>::kBytes;
  static constexpr int TB = 16 / ESZ;       // positions per 16-byte block
  static constexpr int PB = TB / LPC;       // positions of a block finalised by one lane
  static_assert(PB >= 1, "a lane finalises at least one position per block");
  static constexpr int PBYTES = 16 / LPC;   // bytes of those positions
  static constexpr int LC = RB / ESZ;       // positions per chunk
  static constexpr int NBLK = RB / 16;      // 16-byte blocks per row
  static constexpr int NARR = GATE ? 3 : 2; // u, delta (, z)
  // tile bases aligned to the swizzle pattern's period (8 rows of RB bytes)
  static constexpr int ALIGN = 8 * RB;
  static constexpr int pad(int x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }
  static constexpr int TILE = pad(DT * RB);        // one [DT x LC] swizzled tile
  static constexpr int BCT = pad(N * RB);          // one [N x LC] swizzled tile
  static constexpr int STAGE = NARR * TILE + 2 * BCT;
  static constexpr int OFF_STAGES = 0;
  static constexpr int BCF = LC * N * 4;                        // fp32 [LC][N]
  static constexpr int OFF_BCF = OFF_STAGES + S * STAGE;        // [2 buf][B, C]
  // per-warp exchange buffers (LPC > 1): step sizes [32 lanes][PB] and partial
  // contractions [LPC parts][32 lanes][PB]
  static constexpr int XCH_S = 32 * PB;                         // floats
  static constexpr int XCH_WARP = (LPC > 1) ? 4 * (XCH_S + 32 * TB) : 0;
  static constexpr int OFF_XCH = OFF_BCF + 2 * 2 * BCF;
  static constexpr int OFF_BAR = OFF_XCH + WARPS * XCH_WARP;
  static constexpr int SMEM = OFF_BAR + S * 8;
  static constexpr int SMEM_ALLOC = SMEM + ALIGN;               // for base alignment
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
  static constexpr uint32_t TX_BYTES = NARR * DT * RB + 2 * N * RB;
};

struct ChanMaps {
  CUtensorMap u, delta, z, B, C;
};

// Byte offset of 16-byte granule c of row r in a tile of RB-byte rows written by
// TMA with the swizzle of span RB (tile base aligned to 8 * RB): the granule
// index is XOR-ed with address bits 7 and up.
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * RB + ((c ^ (((r * RB) >> 7) & (RB / 16 - 1))) << 4);
}

// widen K io values packed in 32-bit words
template <typename IO, int K>
__device__ __forceinline__ void unpack_words(const uint32_t* w, float* out) {
  if constexpr (sizeof(IO) == 2) {
#pragma unroll
    for (int k = 0; k < K / 2; ++k) {
      out[2 * k] = bf16lo(w[k]);
      out[2 * k + 1] = bf16hi(w[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) out[k] = __uint_as_float(w[k]);
  }
}

// load K consecutive io values (K * size bytes, naturally aligned) from shared memory
template <typename IO, int K>
__device__ __forceinline__ void lds_vals(const uint8_t* p, float* out) {
  constexpr int BYTES = K * sizeof(IO);
  if constexpr (BYTES == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    unpack_words<IO, K>(w, out);
  } else if constexpr (BYTES == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {v.x, v.y};
    unpack_words<IO, K>(w, out);
  } else if constexpr (BYTES == 4) {
    const uint32_t w[1] = {*reinterpret_cast<const uint32_t*>(p)};
    unpack_words<IO, K>(w, out);
  } else {
    static_assert(BYTES == 16 || BYTES == 8 || BYTES == 4, "unsupported vector width");
  }
}

// round K values to io and store them (K * size bytes, naturally aligned)
template <typename IO, int K>
__device__ __forceinline__ void st_vals(void* p, const float* v) {
  constexpr int BYTES = K * sizeof(IO);
  uint32_t w[(BYTES + 3) / 4];
  if constexpr (sizeof(IO) == 2) {
#pragma unroll
    for (int k = 0; k < K / 2; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = __float_as_uint(v[k]);
  }
  if constexpr (BYTES == 16) {
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (BYTES == 8) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else if constexpr (BYTES == 4) {
    *reinterpret_cast<uint32_t*>(p) = w[0];
  } else {
    static_assert(BYTES == 16 || BYTES == 8 || BYTES == 4, "unsupported vector width");
  }
}

// K consecutive floats to / from shared memory (K * 4 bytes, naturally aligned)
template <int K>
__device__ __forceinline__ void st_floats(float* p, const float* v) {
  if constexpr (K == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (K == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  } else {
    static_assert(K == 1, "1, 2 or 4 floats");
    *p = v[0];
  }
}
template <int K>
__device__ __forceinline__ void ld_floats(const float* p, float* v) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int k = 0; k < K; k += 4) {
      const float4 q = *reinterpret_cast<const float4*>(p + k);
      v[k] = q.x; v[k + 1] = q.y; v[k + 2] = q.z; v[k + 3] = q.w;
    }
  } else if constexpr (K == 2) {
    const float2 q = *reinterpret_cast<const float2*>(p);
    v[0] = q.x; v[1] = q.y;
  } else {
    static_assert(K == 1, "1, 2 or a multiple of 4 floats");
    v[0] = *p;
  }
}

// All-gather over the LPC lanes of a channel through this warp's exchange
// buffer: lane `part` holds the PB step sizes of positions [part*PB, part*PB+PB);
// afterwards every lane of the channel holds all TB = LPC*PB in position order.
template <int LPC, int PB>
__device__ __forceinline__ void allgather(const float* mine, float* all, float* xs, int lane) {
  if constexpr (LPC == 1) {
#pragma unroll
    for (int k = 0; k < PB; ++k) all[k] = mine[k];
  } else {
    st_floats<PB>(xs + lane * PB, mine);
    __syncwarp();
    ld_floats<LPC * PB>(xs + (lane & ~(LPC - 1)) * PB, all);
  }
}

// Reduce-scatter over the LPC lanes of a channel: every lane holds partial sums
// for TB positions; afterwards lane `part` holds the full sums of positions
// [part*PB, part*PB + PB).  Each lane writes its partials split by position part
// (row p of the buffer holds every lane's partials for part p), then sums the LPC
// contiguous entries of its channel in row `part`.  The two halves of that read
// are taken in an order that alternates with the part, so that one 16-byte load
// of the warp covers every bank group.
template <int LPC, int TB>
__device__ __forceinline__ void reduce_scatter(const float* v, float* out, float* xp, int lane,
                                               int part) {
  constexpr int PB = TB / LPC;
  if constexpr (LPC == 1) {
#pragma unroll
    for (int k = 0; k < TB; ++k) out[k] = v[k];
  } else {
#pragma unroll
    for (int q = 0; q < LPC; ++q) st_floats<PB>(xp + (q * 32 + lane) * PB, v + q * PB);
    __syncwarp();
    const float* row = xp + (part * 32 + (lane & ~(LPC - 1))) * PB;  // TB floats
    float r[TB];
    if constexpr (TB == 8) {
      const int h = (part & 1) * 4;
      ld_floats<4>(row + h, r);
      ld_floats<4>(row + (4 - h), r + 4);
    } else {
      ld_floats<TB>(row, r);
    }
#pragma unroll
    for (int k = 0; k < PB; ++k) {
      if constexpr (LPC == 4)
        out[k] = (r[k] + r[PB + k]) + (r[2 * PB + k] + r[3 * PB + k]);
      else
        out[k] = r[k] + r[PB + k];
    }
  }
}

// ---------------------------------------------------------------------------
// the state updates and partial contractions of one 16-byte block of positions
// for one lane (its states part*NS .. part*NS + NS - 1).  AR selects the update
// arithmetic: kArFast the fast form Abar (h + w) - w; kArNeg (every A of the channel
// group negative) h + coef (A h + B u) with coef = (2^q - 1) / A from the branch-free
// estimate; kArGen the expm1 series near zero and the dt limit at A == 0.
// ---------------------------------------------------------------------------
template <typename Cfg, bool OUT, int AR>
__device__ __forceinline__ void chan_positions(const float* bcfB, const float* bcfC, int blk,
                                               int part, const float* uj, const float* sj,
                                               const float* Areg, const float* nIA, float* h,
                                               float* acc) {
  constexpr int N = Cfg::N, NS = Cfg::NS, TB = Cfg::TB;
  constexpr bool UACC = AR != kArFast;
#pragma unroll
  for (int j = 0; j < TB; ++j) {
    const int lc = blk * TB + j;  // position within the chunk
    const float dtj = sj[j] * kLn2;  // dt (Euler input term)
    (void)dtj;
    const float* Bp = bcfB + lc * N + part * NS;
    const float* Cp = bcfC + lc * N + part * NS;
    // contraction in a fixed order for every lane split: a packed pair sum per
    // group of 4 states, then a tree over the groups (and over lanes in
    // reduce_scatter), so 1, 2 and 4 lanes per channel give identical bits
    float pg[NS / 4];
#pragma unroll
    for (int m = 0; m < NS; m += 4) {
      f2 a2 = mk2(0.0f, 0.0f);
      const float4 Bv = lds128f(Bp + m);
      const float4 Cv = OUT ? lds128f(Cp + m) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float bv[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
      const float cv[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
#pragma unroll
      for (int pp = 0; pp < 4; pp += 2) {
        const int i = m + pp;
        if constexpr (!UACC) {
          const f2 q = mul2(mk2(sj[j], sj[j]), mk2(Areg[i], Areg[i + 1]));
          const f2 a = mk2(ex2(q.x), ex2(q.y));
          const f2 X = mul2(mk2(bv[pp], bv[pp + 1]), mk2(uj[j], uj[j]));
          f2 hn;
          if constexpr (Cfg::EULER) {
            const f2 W = mul2(X, mk2(dtj, dtj));                // dt B u
            hn = fma2(a, mk2(h[i], h[i + 1]), W);               // Abar h + dt B u
          } else {
            const f2 nw = mul2(X, mk2(nIA[i], nIA[i + 1]));     // -w = -B u / A
            const f2 t = sub2(mk2(h[i], h[i + 1]), nw);         // h + w
            hn = fma2(a, t, nw);                                // Abar (h + w) - w
          }
          h[i] = hn.x;
          h[i + 1] = hn.y;
        } else if constexpr (AR == kArNeg && !Cfg::EULER) {
          // h + (2^q - 1) / A (A h + B u) = Abar h + coef B u; with nq = -q and
          // 1 - 2^q from its branch-free estimate, coef = (1 - 2^q) (-1 / A)
          const f2 nq = mul2(mk2(-sj[j], -sj[j]), mk2(Areg[i], Areg[i + 1]));
          const f2 a = mk2(ex2(-nq.x), ex2(-nq.y));
          const f2 coef = mul2(one_minus_exp2_neg2(nq, a), mk2(nIA[i], nIA[i + 1]));
          const f2 bu = mul2(mk2(bv[pp], bv[pp + 1]), mk2(uj[j], uj[j]));
          const f2 hh = mk2(h[i], h[i + 1]);
          const f2 hn = fma2(coef, fma2(mk2(Areg[i], Areg[i + 1]), hh, bu), hh);
          h[i] = hn.x;
          h[i + 1] = hn.y;
        } else {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float A0 = Areg[i + e];
            const float q = sj[j] * A0;
            const float ahw = ex2(q);
            const float em1 = exp2m1_accurate(q, ahw);
            const float a = (fabsf(q) < kExpm1SeriesMaxQ) ? 1.0f + em1 : ahw;
            // (Abar - 1) / A, or dt at A == 0
            const float coef =
                (Cfg::EULER || A0 == 0.0f) ? sj[j] * kLn2 : em1 * -nIA[i + e];
            h[i + e] = fmaf(a, h[i + e], coef * (bv[pp + e] * uj[j]));
          }
        }
        if constexpr (OUT) a2 = fma2(mk2(cv[pp], cv[pp + 1]), mk2(h[i], h[i + 1]), a2);
      }
      pg[m / 4] = a2.x + a2.y;
    }
    if constexpr (NS == 16)
      acc[j] = (pg[0] + pg[1]) + (pg[2] + pg[3]);
    else if constexpr (NS == 8)
      acc[j] = pg[0] + pg[1];
    else
      acc[j] = pg[0];
  }
}

// ---------------------------------------------------------------------------
// one chunk of positions for one lane (its channel's row `row` of the tiles,
// its states part*NS .. part*NS + NS - 1).  ACC: accurate arithmetic for the
// whole chunk (fp32 io, or a channel group with small |A|); otherwise each block
// whose raw step argument x2 = (delta + bias) log2 e reaches below `x2_min` (the
// argument whose step gives a state update with |dt A log2 e| = kFastPathMinQ)
// takes the accurate update, the rest the fast one.
// ---------------------------------------------------------------------------
// `yrow`: this lane's channel's row of y (null: no output, or a channel past dim).
template <typename Cfg, typename IO, int MODE, bool ACC, bool TAIL, bool NEG, bool CKPT, bool Y>
__device__ __forceinline__ void chan_chunk(const uint8_t* stage, IO* yrow, const float* bcfB,
                                           const float* bcfC, float* xch, int row, int part,
                                           int lane, int l0, int seqlen, const float* Areg,
                                           const float* nIA, float Dd, float bias2, int softplus,
                                           float x2_min, float* h, float& ssum, float* ck,
                                           int64_t ck_stride) {
  constexpr bool OUT = MODE != kModeStates && Y;  // this pass writes y
  constexpr int LPC = Cfg::LPC, TB = Cfg::TB, PB = Cfg::PB, RB = Cfg::RB;
  const uint8_t* tu = stage;
  const uint8_t* td = stage + Cfg::TILE;
  const uint8_t* tz = stage + 2 * Cfg::TILE;
  const int pofs = part * Cfg::PBYTES;

#pragma unroll 1
  for (int blk = 0; blk < Cfg::NBLK; ++blk) {
    const uint32_t off = swz<RB>(row, blk);
    // training forward: the state entering this block, when it starts a checkpoint block
    if (CKPT && ck) {
      const int l = l0 + blk * TB;
      if (l % kCkptPos == 0 && l < seqlen) {
        float* dst = ck + static_cast<int64_t>(l / kCkptPos) * ck_stride;
#pragma unroll
        for (int i = 0; i < Cfg::NS; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(h[i], h[i + 1], h[i + 2], h[i + 3]);
      }
    }
    float uj[TB], sj[TB];
    lds_vals<IO, TB>(tu + off, uj);
    // step sizes of this lane's positions, then shared with the channel's lanes; the
    // smallest raw argument x2 of the block (softplus is monotone) for the choice of
    // update below, formed beside the softplus chain rather than after it
    float x2min;
    {
      float dm[PB], sm[PB];
      lds_vals<IO, PB>(td + off + pofs, dm);
      float x2s[PB];
#pragma unroll
      for (int k = 0; k < PB; ++k) x2s[k] = fmaf(dm[k], kLog2e, bias2);
      x2min = x2s[0];
#pragma unroll
      for (int k = 1; k < PB; ++k) x2min = fminf(x2min, x2s[k]);
#pragma unroll
      for (int k = 0; k < PB; ++k) {
        const float x2 = x2s[k];
        float s = softplus ? (ACC ? softplus_log2_accurate(x2) : softplus_log2_fast(x2)) : x2;
        if constexpr (TAIL) s = (l0 + blk * TB + part * PB + k < seqlen) ? s : 0.0f;  // Abar = 1
        sm[k] = s;
      }
      allgather<LPC, PB>(sm, sj, xch, lane);
      if constexpr (LPC >= 2) x2min = fminf(x2min, __shfl_xor_sync(0xffffffffu, x2min, 1));
      if constexpr (LPC >= 4) x2min = fminf(x2min, __shfl_xor_sync(0xffffffffu, x2min, 2));
    }
    if constexpr (MODE == kModeStates) {
#pragma unroll
      for (int j = 0; j < TB; ++j) ssum += sj[j];
    }
    float acc[TB];
    constexpr int AR_ACC = NEG ? kArNeg : kArGen;
    if constexpr (ACC || Cfg::EULER) {
      // the Euler input term dt B u has no cancellation: the fast form holds for any dt
      chan_positions<Cfg, OUT, ACC ? AR_ACC : kArFast>(bcfB, bcfC, blk, part, uj, sj, Areg, nIA,
                                                       h, acc);
    } else {
      // a step too small for Abar (h + w) - w (its error relative to the update grows
      // like 2^-22 / |q|): this block takes the accurate update.  The decision depends
      // only on the channel's own raw steps and A row, so every lane split takes it
      // alike.  (Past the end of the sequence u is zero-filled, so the fast form
      // leaves h exactly unchanged there whatever is decided.)
      if (!(x2min >= x2_min))
        chan_positions<Cfg, OUT, AR_ACC>(bcfB, bcfC, blk, part, uj, sj, Areg, nIA, h, acc);
      else
        chan_positions<Cfg, OUT, kArFast>(bcfB, bcfC, blk, part, uj, sj, Areg, nIA, h, acc);
    }
    if constexpr (!OUT) continue;
    // full contraction of this lane's positions, then D skip, gate, rounding
    float ym[PB];
    reduce_scatter<LPC, TB>(acc, ym, xch + Cfg::XCH_S, lane, part);
    float um[PB];
    if constexpr (LPC == 1) {
#pragma unroll
      for (int k = 0; k < PB; ++k) um[k] = uj[k];
    } else {
      lds_vals<IO, PB>(tu + off + pofs, um);
    }
#pragma unroll
    for (int k = 0; k < PB; ++k) ym[k] = fmaf(Dd, um[k], ym[k]);
    if constexpr (Cfg::GATE) {
      float zm[PB];
      lds_vals<IO, PB>(tz + off + pofs, zm);
      if constexpr (ACC) {
#pragma unroll
        for (int k = 0; k < PB; ++k) ym[k] *= silu_accurate(zm[k]);
      } else if constexpr (PB % 2 == 0) {
        // y silu(z) = g + g tanh(h) with h = z / 2, g = y h (the hardware tanh), in
        // packed pairs: the same operations as the scalar form below
#pragma unroll
        for (int k = 0; k < PB; k += 2) {
          const f2 h = mul2(mk2(zm[k], zm[k + 1]), mk2(0.5f, 0.5f));
          const f2 g = mul2(mk2(ym[k], ym[k + 1]), h);
          const f2 r = fma2(g, mk2(tanh_hw(h.x), tanh_hw(h.y)), g);
          ym[k] = r.x;
          ym[k + 1] = r.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < PB; ++k) {
          const float h = zm[k] * 0.5f, g = ym[k] * h;
          ym[k] = fmaf(g, tanh_hw(h), g);
        }
      }
    }
    // (the row length is a multiple of the block, as the TMA row pitch requires, so a
    // block lies wholly inside the sequence or wholly past it)
    const int lb = l0 + blk * TB;
    if (yrow != nullptr && (!TAIL || lb < seqlen)) st_vals<IO, PB>(yrow + lb + part * PB, ym);
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// One CTA's work: channels d0 .. d0 + DT - 1 of batch row b over segment `seg`
// (the whole sequence when nseg == 1).  `maps` must live in kernel parameter
// space (a __grid_constant__ argument): TMA reads the descriptors from there.
// CKPT: the training forward, writing the state entering every kCkptPos positions to
// p.ckpt (compiled apart, so that the plain forward carries none of it); Y: the pass
// writes y (a checkpoint-only pass reads neither C nor z and writes no output)
template <typename IO, typename Cfg, int MODE, bool CKPT, bool Y>
__device__ __forceinline__ void channel_body(const ChanMaps& maps, const ScanParams& p, int b,
                                             int d0, int seg, uint8_t* smem_raw) {
  constexpr int N = Cfg::N, NS = Cfg::NS, S = Cfg::S, LC = Cfg::LC;
  constexpr bool OUT = MODE != kModeStates && Y;
  static_assert(Y || CKPT, "a pass writes y, checkpoints or both");
  // bytes one chunk brings in: a pass without output needs u, delta and B only
  constexpr uint32_t TX = OUT ? Cfg::TX_BYTES : 2 * Cfg::DT * Cfg::RB + N * Cfg::RB;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + Cfg::ALIGN - 1) &
      ~static_cast<uintptr_t>(Cfg::ALIGN - 1));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

  const int tid = threadIdx.x;
  const int l_begin = seg * p.seg_len;
  const int l_end = (p.seqlen - l_begin < p.seg_len) ? p.seqlen : l_begin + p.seg_len;
  const int row = tid / Cfg::LPC;
  const int part = tid % Cfg::LPC;
  const int lane = tid & 31;
  float* xch = reinterpret_cast<float*>(smem + Cfg::OFF_XCH + (tid >> 5) * Cfg::XCH_WARP);
  const int d = d0 + row;
  const bool valid = d < p.dim;
  const int nchunks = (l_end - l_begin + LC - 1) / LC;

  // per-lane parameters and state: states part*NS .. part*NS + NS - 1
  float Areg[NS], nIA[NS], h[NS];
  const int64_t state0 = (static_cast<int64_t>(b) * p.dim + d) * N + part * NS;
  // this lane's checkpoint slot (pass 1 of the segmented scan runs from a zero state:
  // it writes none)
  static_assert(!(CKPT && MODE == kModeStates), "the states pass writes no checkpoints");
  float* const ck = (CKPT && valid) ? p.ckpt + state0 : nullptr;
  IO* const yrow = (OUT && valid)
                       ? static_cast<IO*>(p.y) + (static_cast<int64_t>(b) * p.dim + d) * p.seqlen
                       : nullptr;
  const int64_t ck_stride = static_cast<int64_t>(p.batch) * p.dim * N;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float a = valid ? __ldg(p.A + static_cast<int64_t>(d) * N + part * NS + i) : -1.0f;
    Areg[i] = a;
    nIA[i] = (a == 0.0f) ? 0.0f : -1.0f / a;
    h[i] = (MODE != kModeStates && valid && p.h0) ? __ldg(p.h0 + state0 + i) : 0.0f;
  }
  if constexpr (MODE == kModeCarry) {
    // state entering this segment: fold in each earlier segment j as
    // h <- 2^(A * sum_j) h + E_j (the recurrence is linear in h; 2^(A sum_j) is the
    // product of the segment's Abar factors)
    const int64_t chan = static_cast<int64_t>(b) * p.dim + d;
    const int64_t per_seg = static_cast<int64_t>(p.batch) * p.dim;
    if (valid) {
#pragma unroll 1
      for (int j = 0; j < seg; ++j) {
        const float sum = __ldg(p.seg_sum + j * per_seg + chan);
        const float* E = p.seg_state + (j * per_seg + chan) * N + part * NS;
#pragma unroll
        for (int i = 0; i < NS; ++i) h[i] = fmaf(ex2(Areg[i] * sum), h[i], __ldg(E + i));
      }
    }
  }
  float ssum = 0.0f;  // pass 1: sum of the segment's step sizes (log2 units)
  const float Dd = (valid && p.D) ? __ldg(p.D + d) : 0.0f;
  const float bias2 = (valid && p.bias) ? __ldg(p.bias + d) * kLog2e : 0.0f;
  // fast or accurate arithmetic, decided per aligned group of 32 channels (every
  // warp of every lane split lies inside one group, so a channel's arithmetic does
  // not depend on the split): accurate when any |A| of the group is below 1/8; the
  // accurate update without branches when every A of the group is negative
  bool accurate = true, neg = true;
  {
    const int dg = (d0 + (tid >> 5) * (32 / Cfg::LPC)) / 32 * 32 + lane;  // lane's channel
    bool small_a = false, nonneg = false;
    if (dg < p.dim) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const float a = __ldg(p.A + static_cast<int64_t>(dg) * N + i);
        small_a |= !(fabsf(a) >= kFastPathMinAbsA);
        nonneg |= !(a < 0.0f);
      }
    }
    if constexpr (sizeof(IO) == 2) accurate = __any_sync(0xffffffffu, small_a);
    neg = !__any_sync(0xffffffffu, nonneg);
  }
  // smallest raw step argument x2 = (delta + bias) log2 e the fast update takes for
  // this channel: every state's |q| = s |A| must reach kFastPathMinQ, with the step
  // s = log2(1 + 2^x2) (softplus) or s = x2; inverted, x2 = log2(2^s - 1)
  float x2_min = -3.0e38f;
  if (sizeof(IO) == 2 && !accurate && valid) {
    float amin = fabsf(__ldg(p.A + static_cast<int64_t>(d) * N));
#pragma unroll
    for (int i = 1; i < N; ++i) amin = fminf(amin, fabsf(__ldg(p.A + static_cast<int64_t>(d) * N + i)));
    const float s_min = kFastPathMinQ / amin;
    x2_min = p.softplus ? log2f(expm1f(s_min * kLn2)) : s_min;
  }

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.delta);
    prefetch_tmap(&maps.B);
    prefetch_tmap(&maps.C);
    if (Cfg::GATE) prefetch_tmap(&maps.z);
  }
  __syncthreads();

  auto issue_loads = [&](int k) {
    uint8_t* st = smem + Cfg::OFF_STAGES + (k % S) * Cfg::STAGE;
    uint64_t* bar = &full[k % S];
    mbar_arrive_expect_tx(bar, TX);
    const int l = l_begin + k * LC;
    tma_load_3d(st, &maps.u, bar, l, d0, b);
    tma_load_3d(st + Cfg::TILE, &maps.delta, bar, l, d0, b);
    if (Cfg::GATE && OUT) tma_load_3d(st + 2 * Cfg::TILE, &maps.z, bar, l, d0, b);
    tma_load_3d(st + Cfg::NARR * Cfg::TILE, &maps.B, bar, l, 0, b);
    if (OUT) tma_load_3d(st + Cfg::NARR * Cfg::TILE + Cfg::BCT, &maps.C, bar, l, 0, b);
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
    if (arrived) {
      float* bf = reinterpret_cast<float*>(smem + Cfg::OFF_BCF + (k & 1) * 2 * Cfg::BCF);
      const uint8_t* raw = st + Cfg::NARR * Cfg::TILE;
#pragma unroll 1
      for (int piece = tid; piece < (OUT ? 2 : 1) * N * Cfg::NBLK; piece += Cfg::THREADS) {
        const int arr = piece / (N * Cfg::NBLK);
        const int rem = piece % (N * Cfg::NBLK);
        const int n = rem % N, kb = rem / N;
        float v[Cfg::TB];
        lds_vals<IO, Cfg::TB>(raw + arr * Cfg::BCT + swz<Cfg::RB>(n, kb), v);
        float* dst = bf + arr * (Cfg::BCF / 4) + (kb * Cfg::TB) * N + n;
#pragma unroll
        for (int e = 0; e < Cfg::TB; ++e) dst[e * N] = v[e];
      }
    }
    if (__syncthreads_or(!arrived)) {
      ok = false;
      break;
    }
    if (tid == 0 && k >= 1 && k - 1 + S < nchunks) {
      fence_proxy_async_smem();
      issue_loads(k - 1 + S);  // stage of chunk k-1 is free: every thread passed the barrier
      ++issued;
    }
    const float* bcfB =
        reinterpret_cast<const float*>(smem + Cfg::OFF_BCF + (k & 1) * 2 * Cfg::BCF);
    const float* bcfC = bcfB + Cfg::BCF / 4;
    const int l0 = l_begin + k * LC;
    const bool tail = l0 + LC > p.seqlen;
    // (the group flags are warp-uniform: every lane of a warp takes the same branch)
#define SSM_CHAN_CHUNK(ACC, TAIL, NEG)                                                        \
  chan_chunk<Cfg, IO, MODE, ACC, TAIL, NEG, CKPT, Y>(st, yrow, bcfB, bcfC, xch, row, part, lane, \
                                                     l0, p.seqlen, Areg, nIA, Dd, bias2,        \
                                                     p.softplus, x2_min, h, ssum, ck, ck_stride)
    bool fast_chunk = false;
    if constexpr (sizeof(IO) == 2) fast_chunk = !accurate;
    if (fast_chunk) {
      if constexpr (sizeof(IO) == 2) {
        if (neg) {
          if (!tail) SSM_CHAN_CHUNK(false, false, true); else SSM_CHAN_CHUNK(false, true, true);
        } else {
          if (!tail) SSM_CHAN_CHUNK(false, false, false); else SSM_CHAN_CHUNK(false, true, false);
        }
      }
    } else {
      if (neg) SSM_CHAN_CHUNK(true, true, true); else SSM_CHAN_CHUNK(true, true, false);
    }
#undef SSM_CHAN_CHUNK
  }
  __syncthreads();
  if (tid == 0) {
    if (!ok) {
      // a wait gave up at chunk k: before the CTA exits, wait (bounded) for every
      // load that may still be in flight into the ring (chunks k .. issued-1)
      for (int kk = k; kk < issued; ++kk) (void)mbar_wait_bounded(&full[kk % S], (kk / S) & 1);
    }
  }
  if (ok && valid) {
    if constexpr (MODE == kModeStates) {
      const int64_t chan = static_cast<int64_t>(b) * p.dim + d;
      const int64_t per_seg = static_cast<int64_t>(p.batch) * p.dim;
      float* E = p.seg_state + (seg * per_seg + chan) * N + part * NS;
#pragma unroll
      for (int i = 0; i < NS; ++i) E[i] = h[i];
      if (part == 0) p.seg_sum[seg * per_seg + chan] = ssum;
    } else if (p.h_last && seg == p.nseg - 1) {
#pragma unroll
      for (int i = 0; i < NS; ++i) p.h_last[state0 + i] = h[i];
    }
  }
}

template <typename IO, typename Cfg, int MODE, bool CKPT = false, bool Y = true>
__global__ void __launch_bounds__(Cfg::THREADS)
    scan_channel_kernel(const __grid_constant__ ChanMaps maps, const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  // block index = (segment * batch + b) * dtiles + channel tile
  const int rest = blockIdx.x / p.dtiles;
  channel_body<IO, Cfg, MODE, CKPT, Y>(maps, p, rest % p.batch, (blockIdx.x % p.dtiles) * Cfg::DT,
                              rest / p.batch, smem_raw);
}

// ---------------------------------------------------------------------------
// mixed split: whole SMs' worth of one-lane-per-channel CTAs plus the remainder
// in four-lanes-per-channel CTAs
// ---------------------------------------------------------------------------
// With T 128-channel tiles on `sms` SMs, one lane per channel runs T / sms CTAs
// per SM when that divides; otherwise the SMs that get one more CTA set the time.
// The mixed launch gives every SM exactly k = floor(T / sms) one-lane CTAs (CfgA)
// and splits the other T - k * sms tiles into 32-channel CTAs with four lanes per
// channel (CfgB), which spread over the SMs at a quarter of the cost each.  The
// block scheduler does not guarantee k CTAs per SM, so each CTA picks its role
// when it starts: the first k CTAs to arrive on an SM take whole tiles, the
// others take quarter tiles (each falls back to the other pool when its own is
// empty; there are exactly as many CTAs as units).  1 and 4 lanes per channel
// give identical bits, so the outcome does not depend on the assignment.
struct MixSched {
  int k;               // one-lane CTAs per SM
  int n_tiles;         // whole tiles for CfgA: tiles 0 .. n_tiles - 1 (b-major)
  int n_quarters;      // quarter tiles for CfgB: quarters of tiles n_tiles .. T - 1
  int dtiles128;       // 128-channel tiles per batch row
  unsigned* counters;  // [0] next whole tile, [1] next quarter, [2 + smid] arrivals
  unsigned max_sm_slots;  // SM ids with an arrival counter
};

template <typename IO, typename CfgA, typename CfgB, bool CKPT = false, bool Y = true>
__global__ void __launch_bounds__(CfgA::THREADS)
    scan_channel_mixed_kernel(const __grid_constant__ ChanMaps mapsA,
                              const __grid_constant__ ChanMaps mapsB, const ScanParams p,
                              const MixSched m) {
  static_assert(CfgA::THREADS == CfgB::THREADS, "one block shape for both roles");
  extern __shared__ uint8_t smem_raw[];
  __shared__ int role_unit[2];
  if (threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const int arrival = (smid < m.max_sm_slots)
                            ? static_cast<int>(atomicAdd(&m.counters[2 + smid], 1u))
                            : m.k;  // no counter for this SM: take quarter tiles
    int role = -1, unit = 0;
    if (arrival < m.k) {
      const int t = static_cast<int>(atomicAdd(&m.counters[0], 1u));
      if (t < m.n_tiles) role = 0, unit = t;
    }
    if (role < 0) {
      const int q = static_cast<int>(atomicAdd(&m.counters[1], 1u));
      if (q < m.n_quarters) role = 1, unit = q;
    }
    if (role < 0) {
      const int t = static_cast<int>(atomicAdd(&m.counters[0], 1u));
      if (t < m.n_tiles) role = 0, unit = t;
    }
    role_unit[0] = role;
    role_unit[1] = unit;
  }
  __syncthreads();
  const int role = role_unit[0], unit = role_unit[1];
  if (role == 0) {
    channel_body<IO, CfgA, kModeFull, CKPT, Y>(mapsA, p, unit / m.dtiles128,
                                               (unit % m.dtiles128) * 128, 0, smem_raw);
  } else if (role == 1) {
    const int tile = m.n_tiles + unit / 4;
    const int d0 = (tile % m.dtiles128) * 128 + (unit % 4) * 32;
    if (d0 < p.dim)
      channel_body<IO, CfgB, kModeFull, CKPT, Y>(mapsB, p, tile / m.dtiles128, d0, 0, smem_raw);
  }
}

}  // namespace ssm
