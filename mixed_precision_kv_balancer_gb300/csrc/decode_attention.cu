// K7 + K8: decode attention over the two-tier mixed-precision cache.
//
// Sources: "No Token Left Behind" reading notes (velog), section 3.4
// "Accelerating the Mixed-Precision KV Cache" and the paperlayer summary,
// section 3.4 (attention is permutation invariant after positional embedding,
// so each precision is a contiguous tier; K and V are low precision while Q and
// the attention map stay floating point; decode is memory bound); notes "2)
// Outlier-aware handling" (quantised keys hold I(k*b) and are attended with
// q/b).
//
// Design (split-K flash decoding, one pass over the packed cache):
// * Grid (splits, B*Hkv).  A CTA owns a contiguous chunk of ONE tier of one
//   (batch, key head); its 4 warps stream stages of that chunk through private
//   shared-memory rings filled by 16-byte cp.async (zero-filled past the end).
// * Every query head of the key head's group is served by the same pass: the
//   group is the mma's N dimension, so the cache is read once per key head.
// * QK^T: m16n8k16 with 16 tokens as M and the columns (head, hi|lo) as N.  The
//   query is carried as two fp16 parts (hi = fp16(q), lo = fp16(q - hi)) in the
//   two columns of its head, giving ~22-bit query precision for free on N = 8.
// * Quantised tiers: codes enter the mma as exact fp16 integers (code | 0x6400
//   minus 1024), one accumulator per 64-channel group, and the scale/zero are
//   applied afterwards per token and group:
//     q.k~ = s0 * (q.c)_g0 + s1 * (q.c)_g1 + z0 * sum_g0(q) + z1 * sum_g1(q).
//   Channel order inside a group is permuted to whatever the bit unpacking
//   yields; the query fragments use the same permutation.
// * PV: o^T = V^T P^T with channels as M, tokens as K and (head, hi|lo) as N;
//   P (times the value scale of the group, for quantised tiers) is split into
//   fp16 hi/lo parts and moved from the accumulator layout into the operand
//   layout with movmatrix; the value zero-point term sum_i p_i z_i is kept in
//   fp32 registers.
// * Online softmax in base 2 per stage; the CTA merges its warps and writes one
//   (m, l, o) partial per head; K8 merges the partials of both tiers.
// Roofline: HBM-bound; the algorithmic bytes are the packed cache rows
// (512 / 272 / 144 / 80 B per token and key head for FP16 / INT8 / INT4 / INT2).
#include <algorithm>

#include "common.cuh"

namespace mikv {
int validate_cache_public(const mikv_cache* c, const char* who);

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;        // ring depth per warp
constexpr float kLog2e = 1.4426950408889634f;

template <int BITS>
struct Fmt {
  static constexpr bool kQuant = BITS != 16;
  static constexpr int kRB = kD * BITS / 8;                        // bytes per token row
  static constexpr int kST = BITS == 16 ? 16 : (BITS == 8 ? 32 : 64);  // tokens per stage
  static constexpr int kMetaB = kQuant ? 8 : 0;                    // (scale, zero) x 2 groups
  static constexpr int kStageBytes = kST * (2 * kRB + 2 * kMetaB);
  static constexpr int kOffV = kST * kRB;
  static constexpr int kOffKM = 2 * kST * kRB;
  static constexpr int kOffVM = 2 * kST * kRB + kST * kMetaB;
};

struct TierPtrs {
  const uint8_t* k;
  const uint8_t* v;
  const uint8_t* km;  // meta rows of 8 bytes (quantised tiers)
  const uint8_t* vm;
  int cap, n;
};

struct Params {
  const __half* q;     // [B][Hq][D]
  const float* bal;    // [B][Hkv][D] or null
  TierPtrs hi, lo;
  int Hq, Hkv, rep;
  int chunk_hi, chunk_lo;  // tokens per CTA
  int nsplit_hi;           // splits [0, nsplit_hi) are hi-tier CTAs
  int smax;                // split stride of the workspace
  float* hi_logits;        // [B][Hq][cap_hi] or null
  float* ws_o;             // [B*Hq][smax][D]
  float* ws_ml;            // [B*Hq][smax][2]
};

// ---------------------------------------------------------------------------------
// stage loads
template <int BITS>
__device__ __forceinline__ void load_stage(uint32_t sb, const TierPtrs& t, long row0, int nvalid,
                                           int lane) {
  using F = Fmt<BITS>;
  constexpr int kChunksPerRow = F::kRB / 16;
  constexpr int kChunks = F::kST * kChunksPerRow;
#pragma unroll
  for (int i = lane; i < kChunks; i += 32) {
    const int r = i / kChunksPerRow, cc = i % kChunksPerRow;
    const bool ok = r < nvalid;
    uint32_t off;
    if constexpr (BITS == 16) off = r * F::kRB + ((cc ^ (r & 7)) << 4);  // 128B-swizzled rows
    else off = i * 16;
    const long g = ok ? (row0 + r) * F::kRB + cc * 16 : 0;
    cp_async16(sb + off, t.k + g, ok);
    cp_async16(sb + F::kOffV + off, t.v + g, ok);
  }
  if constexpr (F::kQuant) {
#pragma unroll
    for (int r = lane; r < F::kST; r += 32) {
      const bool ok = r < nvalid;
      const long g = ok ? (row0 + r) * 8 : 0;
      cp_async8(sb + F::kOffKM + r * 8, t.km + g, ok);
      cp_async8(sb + F::kOffVM + r * 8, t.vm + g, ok);
    }
  }
}

// ---------------------------------------------------------------------------------
// unpacking: codes -> fp16 pairs holding exact integers
__device__ __forceinline__ uint32_t fix1024(uint32_t bits_with_magic) {
  __half2 h = *reinterpret_cast<__half2*>(&bits_with_magic);
  h = __hsub2(h, __half2half2(__ushort_as_half(0x6400)));
  return *reinterpret_cast<uint32_t*>(&h);
}

// K side: the 16 channels [gr*64 + tig*16, +16) of one token row -> 8 pairs.
// Pair p holds local channels (ca(p), cb(p)) in its (low, high) halves.
template <int BITS>
__device__ __forceinline__ void unpack_k16(uint32_t srow, int gr, int tig, uint32_t (&pr)[8]) {
  if constexpr (BITS == 2) {
    const uint32_t w = lds32(srow + gr * 16 + tig * 4);
#pragma unroll
    for (int p = 0; p < 8; ++p) pr[p] = fix1024(((w >> (2 * p)) & 0x00030003u) | 0x64006400u);
  } else if constexpr (BITS == 4) {
    const uint2 w = lds64(srow + gr * 32 + tig * 8);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      pr[p] = fix1024(((w.x >> (4 * p)) & 0x000F000Fu) | 0x64006400u);
      pr[p + 4] = fix1024(((w.y >> (4 * p)) & 0x000F000Fu) | 0x64006400u);
    }
  } else {
    const uint4 w = lds128(srow + gr * 64 + tig * 16);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pr[2 * i] = fix1024(__byte_perm(ww[i], 0x64u, 0x4140));
      pr[2 * i + 1] = fix1024(__byte_perm(ww[i], 0x64u, 0x4342));
    }
  }
}
template <int BITS>
__host__ __device__ constexpr int k_ca(int p) {
  return BITS == 2 ? p : (BITS == 4 ? (p < 4 ? p : p + 4) : 2 * p);
}
template <int BITS>
__host__ __device__ constexpr int k_cb(int p) {
  return BITS == 2 ? p + 8 : (BITS == 4 ? (p < 4 ? p + 4 : p + 8) : 2 * p + 1);
}

// V side: the 8 channels [gr*64 + gid*8, +8) of two tokens (ta, tb) -> 8 pairs,
// pair c = (code[ta][c], code[tb][c]).
template <int BITS>
__device__ __forceinline__ void unpack_v8(uint32_t sa, uint32_t sb_, int gr, int gid,
                                          uint32_t (&pr)[8]) {
  if constexpr (BITS == 2) {
    const uint32_t ua = lds16(sa + gr * 16 + gid * 2), ub = lds16(sb_ + gr * 16 + gid * 2);
    const uint32_t w = ua | (ub << 16);
#pragma unroll
    for (int c = 0; c < 8; ++c) pr[c] = fix1024(((w >> (2 * c)) & 0x00030003u) | 0x64006400u);
  } else if constexpr (BITS == 4) {
    const uint32_t ua = lds32(sa + gr * 32 + gid * 4), ub = lds32(sb_ + gr * 32 + gid * 4);
    const uint32_t wl = __byte_perm(ua, ub, 0x5410), wh = __byte_perm(ua, ub, 0x7632);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      pr[c] = fix1024(((wl >> (4 * c)) & 0x000F000Fu) | 0x64006400u);
      pr[c + 4] = fix1024(((wh >> (4 * c)) & 0x000F000Fu) | 0x64006400u);
    }
  } else {
    const uint2 ua = lds64(sa + gr * 64 + gid * 8), ub = lds64(sb_ + gr * 64 + gid * 8);
    const uint32_t t0 = __byte_perm(ua.x, ub.x, 0x5140), t1 = __byte_perm(ua.x, ub.x, 0x7362);
    const uint32_t t2 = __byte_perm(ua.y, ub.y, 0x5140), t3 = __byte_perm(ua.y, ub.y, 0x7362);
    pr[0] = fix1024(__byte_perm(t0, 0x64u, 0x4140));
    pr[1] = fix1024(__byte_perm(t0, 0x64u, 0x4342));
    pr[2] = fix1024(__byte_perm(t1, 0x64u, 0x4140));
    pr[3] = fix1024(__byte_perm(t1, 0x64u, 0x4342));
    pr[4] = fix1024(__byte_perm(t2, 0x64u, 0x4140));
    pr[5] = fix1024(__byte_perm(t2, 0x64u, 0x4342));
    pr[6] = fix1024(__byte_perm(t3, 0x64u, 0x4140));
    pr[7] = fix1024(__byte_perm(t3, 0x64u, 0x4342));
  }
}

// ---------------------------------------------------------------------------------
template <int NT>
struct State {
  float m[NT];          // running max (base-2 logits), uniform over the 8 lanes of a head
  float l[NT];          // per-lane partial denominator
  float zs[NT][2];      // per-lane partial sum_i p_i * zero_v,i per value group
  float o[NT][8][4];    // PV accumulators: 8 channel tiles x (2 rows x (hi, lo))
};

// One stage of BITS-format tokens for one warp.
template <int BITS, int NT>
__device__ __forceinline__ void compute_stage(uint32_t sb, int nvalid, const uint32_t (&bq)[NT][8][2],
                                              const float (&qsum)[NT][2], State<NT>& st,
                                              float* logit_out, int logit_stride, int rep,
                                              int lane) {
  using F = Fmt<BITS>;
  constexpr int kSub = F::kST / 16;
  const int gid = lane >> 2, tig = lane & 3;
  const float kScale = rsqrtf(static_cast<float>(kD));  // 1/sqrt(128), exact power-of-two root
  float x[kSub][NT][2];  // base-2 logits of rows gid, gid+8

  // ---- QK^T for every 16-token sub-tile of the stage
#pragma unroll
  for (int sub = 0; sub < kSub; ++sub) {
    const int r0 = sub * 16;
    if constexpr (!F::kQuant) {
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chunk = 2 * s + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sb + row * F::kRB + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma16816(acc[t], a0, a1, a2, a3, bq[t][s][0], bq[t][s][1]);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        x[sub][t][0] = (acc[t][0] + acc[t][1]) * kScale;
        x[sub][t][1] = (acc[t][2] + acc[t][3]) * kScale;
      }
    } else {
      float acc[NT][2][4];
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int gr = 0; gr < 2; ++gr) acc[t][gr][0] = acc[t][gr][1] = acc[t][gr][2] = acc[t][gr][3] = 0.f;
#pragma unroll
      for (int gr = 0; gr < 2; ++gr) {
        uint32_t pa[8], pb[8];
        unpack_k16<BITS>(sb + (r0 + gid) * F::kRB, gr, tig, pa);
        unpack_k16<BITS>(sb + (r0 + gid + 8) * F::kRB, gr, tig, pb);
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            mma16816(acc[t][gr], pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1],
                     bq[t][gr * 4 + s][0], bq[t][gr * 4 + s][1]);
      }
      const uint2 ma = lds64(sb + F::kOffKM + (r0 + gid) * 8);
      const uint2 mb = lds64(sb + F::kOffKM + (r0 + gid + 8) * 8);
      const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&ma.x));
      const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&ma.y));
      const float2 b0 = __half22float2(*reinterpret_cast<const __half2*>(&mb.x));
      const float2 b1 = __half22float2(*reinterpret_cast<const __half2*>(&mb.y));
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float da0 = acc[t][0][0] + acc[t][0][1], da1 = acc[t][1][0] + acc[t][1][1];
        const float db0 = acc[t][0][2] + acc[t][0][3], db1 = acc[t][1][2] + acc[t][1][3];
        x[sub][t][0] = (a0.x * da0 + a1.x * da1 + a0.y * qsum[t][0] + a1.y * qsum[t][1]) * kScale;
        x[sub][t][1] = (b0.x * db0 + b1.x * db1 + b0.y * qsum[t][0] + b1.y * qsum[t][1]) * kScale;
      }
    }
    // natural logits out (important tier) and masking of rows past the end
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int head = t * 4 + tig;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = r0 + gid + 8 * h;
        if (r < nvalid) {
          if (logit_out != nullptr && head < rep) logit_out[head * logit_stride + r] = x[sub][t][h];
          x[sub][t][h] *= kLog2e;
        } else {
          x[sub][t][h] = -INFINITY;
        }
      }
    }
  }

  // ---- online softmax update (one max per stage)
  float mnew[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float mx = -INFINITY;
#pragma unroll
    for (int sub = 0; sub < kSub; ++sub) mx = fmaxf(mx, fmaxf(x[sub][t][0], x[sub][t][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mnew[t] = fmaxf(st.m[t], mx);
    const float alpha = exp2f(st.m[t] - mnew[t]);  // 0 on the first stage (m = -inf)
    st.m[t] = mnew[t];
    st.l[t] *= alpha;
    st.zs[t][0] *= alpha;
    st.zs[t][1] *= alpha;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[t][j][e] *= alpha;
  }

  // ---- P V for every sub-tile
#pragma unroll
  for (int sub = 0; sub < kSub; ++sub) {
    const int r0 = sub * 16;
    float p[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      p[t][0] = exp2f(x[sub][t][0] - mnew[t]);
      p[t][1] = exp2f(x[sub][t][1] - mnew[t]);
      st.l[t] += p[t][0] + p[t][1];
    }
    if constexpr (!F::kQuant) {
      uint32_t bp[NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          __half hi, lo;
          split_f16(p[t][h], hi, lo);
          bp[t][h] = movmatrix_t(pack_half2(hi, lo));
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = 2 * j + ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(sb + F::kOffV + row * F::kRB + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma16816(st.o[t][j], a0, a1, a2, a3, bp[t][0], bp[t][1]);
      }
    } else {
      // value scale/zero of rows gid, gid+8 for both groups
      const uint2 ma = lds64(sb + F::kOffVM + (r0 + gid) * 8);
      const uint2 mb = lds64(sb + F::kOffVM + (r0 + gid + 8) * 8);
      const float2 va[2] = {__half22float2(*reinterpret_cast<const __half2*>(&ma.x)),
                            __half22float2(*reinterpret_cast<const __half2*>(&ma.y))};
      const float2 vb[2] = {__half22float2(*reinterpret_cast<const __half2*>(&mb.x)),
                            __half22float2(*reinterpret_cast<const __half2*>(&mb.y))};
      uint32_t bp[NT][2][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int gr = 0; gr < 2; ++gr) {
          st.zs[t][gr] += p[t][0] * va[gr].y + p[t][1] * vb[gr].y;
          __half hi, lo;
          split_f16(p[t][0] * va[gr].x, hi, lo);
          bp[t][gr][0] = movmatrix_t(pack_half2(hi, lo));
          split_f16(p[t][1] * vb[gr].x, hi, lo);
          bp[t][gr][1] = movmatrix_t(pack_half2(hi, lo));
        }
      }
      const uint32_t s01a = sb + F::kOffV + (r0 + 2 * tig) * F::kRB;
      const uint32_t s01b = s01a + F::kRB;
      const uint32_t s89a = sb + F::kOffV + (r0 + 2 * tig + 8) * F::kRB;
      const uint32_t s89b = s89a + F::kRB;
#pragma unroll
      for (int gr = 0; gr < 2; ++gr) {
        uint32_t v01[8], v89[8];
        unpack_v8<BITS>(s01a, s01b, gr, gid, v01);
        unpack_v8<BITS>(s89a, s89b, gr, gid, v89);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            mma16816(st.o[t][gr * 4 + jj], v01[jj], v01[4 + jj], v89[jj], v89[4 + jj], bp[t][gr][0],
                     bp[t][gr][1]);
      }
    }
  }
}

// Output channel of accumulator row (m-tile j, row gid or gid+8) for a format.
template <int BITS>
__device__ __forceinline__ int out_channel(int j, int gid, int h) {
  if constexpr (BITS == 16) return 16 * j + gid + 8 * h;
  else return (j >> 2) * 64 + gid * 8 + 4 * h + (j & 3);
}

// Build the query fragments of this CTA's tier: columns (head, hi|lo) of n-tile t.
template <int BITS, int NT>
__device__ __forceinline__ void build_q(const float* qs /*smem [8][kD]*/, int rep, int lane,
                                        uint32_t (&bq)[NT][8][2], float (&qsum)[NT][2]) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int head = t * 4 + (gid >> 1);
    const bool part_lo = gid & 1;
    auto val = [&](int c) -> __half {
      const float x = head < rep ? qs[head * kD + c] : 0.f;
      __half hi, lo;
      split_f16(x, hi, lo);
      return part_lo ? lo : hi;
    };
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      int c0, c1, c2, c3;
      if constexpr (BITS == 16) {
        c0 = s * 16 + 2 * tig;
        c1 = c0 + 1;
        c2 = c0 + 8;
        c3 = c0 + 9;
      } else {
        const int gr = s >> 2, sp = s & 3, base = gr * 64 + tig * 16;
        c0 = base + k_ca<BITS>(2 * sp);
        c1 = base + k_cb<BITS>(2 * sp);
        c2 = base + k_ca<BITS>(2 * sp + 1);
        c3 = base + k_cb<BITS>(2 * sp + 1);
      }
      bq[t][s][0] = pack_half2(val(c0), val(c1));
      bq[t][s][1] = pack_half2(val(c2), val(c3));
    }
    // per-group query sums for the zero-point term (thread's own head t*4+tig)
    const int myhead = t * 4 + tig;
#pragma unroll
    for (int gr = 0; gr < 2; ++gr) {
      float sum = 0.f;
      if (myhead < rep)
        for (int c = 0; c < kGS; ++c) sum += qs[myhead * kD + gr * kGS + c];
      qsum[t][gr] = sum;
    }
  }
}

template <int BITS, int NT>
__device__ void run_tier(const Params& P, const TierPtrs& tier, int unit, int split, int chunk,
                         bool is_hi, uint8_t* smem, float* qs) {
  using F = Fmt<BITS>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = unit / P.Hkv, g = unit % P.Hkv;
  const int rep = P.rep;

  // query (balanced for quantised tiers) staged in shared memory as fp32
  for (int i = threadIdx.x; i < 8 * kD; i += kThreads) {
    const int h = i / kD, c = i % kD;
    float x = 0.f;
    if (h < rep) {
      x = __half2float(P.q[(static_cast<long>(b) * P.Hq + g * rep + h) * kD + c]);
      if (F::kQuant && P.bal) x = __fdiv_rn(x, P.bal[static_cast<long>(unit) * kD + c]);
    }
    qs[i] = x;
  }
  __syncthreads();
  uint32_t bq[NT][8][2];
  float qsum[NT][2];
  build_q<BITS, NT>(qs, rep, lane, bq, qsum);

  State<NT> st;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    st.m[t] = -INFINITY;
    st.l[t] = 0.f;
    st.zs[t][0] = st.zs[t][1] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[t][j][e] = 0.f;
  }

  const int t_begin = split * chunk;
  const int t_end = min(tier.n, t_begin + chunk);
  const int nst = (t_end - t_begin + F::kST - 1) / F::kST;   // stages in this CTA
  const long row_base = static_cast<long>(unit) * tier.cap;
  // this warp's ring
  uint8_t* ring = smem + warp * (kStages * F::kStageBytes);
  const uint32_t ring_s = smem_u32(ring);
  float* lrow = nullptr;
  if (is_hi && P.hi_logits)
    lrow = P.hi_logits + (static_cast<long>(b) * P.Hq + g * rep) * tier.cap;

  // warp w handles stages w, w+4, ...
  int issued = 0;
  auto issue = [&](int k) {  // k-th stage of this warp
    const int sidx = warp + k * kWarps;
    if (sidx < nst) {
      const int tok0 = t_begin + sidx * F::kST;
      load_stage<BITS>(ring_s + (k % kStages) * F::kStageBytes, tier, row_base + tok0,
                       min(F::kST, t_end - tok0), lane);
    }
    cp_async_commit();
  };
  for (; issued < kStages - 1; ++issued) issue(issued);
  for (int k = 0; warp + k * kWarps < nst; ++k) {
    issue(issued++);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int tok0 = t_begin + (warp + k * kWarps) * F::kST;
    compute_stage<BITS, NT>(ring_s + (k % kStages) * F::kStageBytes, min(F::kST, t_end - tok0), bq,
                            qsum, st, lrow ? lrow + tok0 : nullptr, tier.cap, rep, lane);
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- CTA merge of the 4 warps' partial states -> one (m, l, o) per head
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float l = st.l[t], z0 = st.zs[t][0], z1 = st.zs[t][1];
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, o);
      z0 += __shfl_xor_sync(0xffffffffu, z0, o);
      z1 += __shfl_xor_sync(0xffffffffu, z1, o);
    }
    st.l[t] = l;
    st.zs[t][0] = z0;
    st.zs[t][1] = z1;
  }
  __syncthreads();  // rings are reused for the merge below
  float* red_o = reinterpret_cast<float*>(smem);                // [kWarps][8 heads][kD]
  float* red_m = red_o + kWarps * 8 * kD;                        // [kWarps][8]
  float* red_l = red_m + kWarps * 8;                             // [kWarps][8]
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int head = t * 4 + tig;
    float* dst = red_o + (warp * 8 + head) * kD;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = out_channel<BITS>(j, gid, h);
        float v = st.o[t][j][2 * h] + st.o[t][j][2 * h + 1];
        if constexpr (F::kQuant) v += (c < kGS) ? st.zs[t][0] : st.zs[t][1];
        dst[c] = v;
      }
    }
    if (gid == 0) {
      red_m[warp * 8 + head] = st.m[t];
      red_l[warp * 8 + head] = st.l[t];
    }
  }
  __syncthreads();
  const int c = threadIdx.x;  // one channel per thread
  const int split_index = is_hi ? split : P.nsplit_hi + split;
  for (int h = 0; h < rep; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_m[w * 8 + h];
      const float sc = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      L += sc * red_l[w * 8 + h];
      O += sc * red_o[(w * 8 + h) * kD + c];
    }
    const long row = (static_cast<long>(b) * P.Hq + g * rep + h) * P.smax + split_index;
    P.ws_o[row * kD + c] = O;
    if (c == 0) {
      P.ws_ml[row * 2] = M;
      P.ws_ml[row * 2 + 1] = L;
    }
  }
}

template <int HI, int LO, int NT>
__global__ void __launch_bounds__(kThreads) decode_partial_kernel(Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float qs[8 * kD];
  const int unit = blockIdx.y;
  const int sx = blockIdx.x;
  if (sx < P.nsplit_hi) run_tier<HI, NT>(P, P.hi, unit, sx, P.chunk_hi, true, smem, qs);
  else run_tier<LO, NT>(P, P.lo, unit, sx - P.nsplit_hi, P.chunk_lo, false, smem, qs);
}

// K8: merge the split partials (base-2 max m, sum l, unnormalised o) of one query head.
__global__ void __launch_bounds__(kD) decode_merge_kernel(const float* __restrict__ ws_o,
                                                          const float* __restrict__ ws_ml,
                                                          int smax, int nsplit,
                                                          float* __restrict__ out,
                                                          float* __restrict__ lse) {
  const int row = blockIdx.x;  // b*Hq + h
  const int c = threadIdx.x;
  const float* ml = ws_ml + static_cast<long>(row) * smax * 2;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[2 * s]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = ml[2 * s];
    const float sc = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
    L += sc * ml[2 * s + 1];
    O += sc * ws_o[(static_cast<long>(row) * smax + s) * kD + c];
  }
  out[static_cast<long>(row) * kD + c] = O / L;
  if (c == 0) lse[row] = (M + log2f(L)) * 0.69314718055994531f;
}

// ---------------------------------------------------------------------------------
// host-side split plan
int stage_tokens(int bits) { return bits == 16 ? 16 : (bits == 8 ? 32 : 64); }
int row_cost(int bits) { return bits == 16 ? 512 : 2 * (kD * bits / 8) + 16; }
int stage_bytes(int bits) { return stage_tokens(bits) * row_cost(bits); }

struct Plan {
  int chunk_hi, chunk_lo, smax_hi, smax_lo;
};

Plan make_plan(const mikv_cache* c) {
  // chunk sizes from the capacities, so the workspace fits every count <= capacity
  const double units = static_cast<double>(c->B) * c->Hkv;
  const double total = units * (static_cast<double>(c->cap_hi) * row_cost(c->hi_bits) +
                                 static_cast<double>(c->cap_lo) * row_cost(c->lo_bits));
  double target = total / (kNumSMs * 2.0 * 6.0);       // ~6 waves of 2 CTAs per SM
  target = std::min(std::max(target, 16.0 * 1024), 192.0 * 1024);
  auto chunk_for = [&](int bits) {
    int per_warp = static_cast<int>(target / (kWarps * stage_bytes(bits)) + 0.5);
    per_warp = std::max(per_warp, 1);
    return per_warp * kWarps * stage_tokens(bits);
  };
  Plan p;
  p.chunk_hi = chunk_for(c->hi_bits);
  p.chunk_lo = chunk_for(c->lo_bits);
  p.smax_hi = (c->cap_hi + p.chunk_hi - 1) / p.chunk_hi;
  p.smax_lo = (c->cap_lo + p.chunk_lo - 1) / p.chunk_lo;
  return p;
}

template <int HI, int LO, int NT>
int launch(const Params& P, dim3 grid, cudaStream_t s) {
  const int smem = kWarps * kStages * std::max(Fmt<HI>::kStageBytes, Fmt<LO>::kStageBytes);
  auto kern = decode_partial_kernel<HI, LO, NT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("decode_partial_kernel attribute");
  kern<<<grid, kThreads, smem, s>>>(P);
  return check_launch("decode_partial_kernel");
}

template <int HI, int LO>
int launch_nt(const Params& P, dim3 grid, cudaStream_t s) {
  return P.rep <= 4 ? launch<HI, LO, 1>(P, grid, s) : launch<HI, LO, 2>(P, grid, s);
}

}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" size_t mikv_decode_workspace_bytes(const mikv_cache* c) {
  if (validate_cache_public(c, "decode_workspace_bytes") != MIKV_OK) return 0;
  const Plan p = make_plan(c);
  const size_t rows = static_cast<size_t>(c->B) * c->Hq * (p.smax_hi + p.smax_lo);
  return align_up(rows * kD * sizeof(float), 256) + align_up(rows * 2 * sizeof(float), 256);
}

extern "C" int mikv_decode_attention(const uint16_t* q, const mikv_cache* c, float* out,
                                     float* lse, float* hi_logits, void* ws, size_t ws_bytes,
                                     void* stream) {
  clear_error();
  if (int e = validate_cache_public(c, "decode_attention")) return e;
  if (!q || !out || !lse || !ws) return fail(MIKV_EINVAL, "decode_attention: null pointer");
  if (c->n_hi + c->n_lo < 1) return fail(MIKV_ESHAPE, "decode_attention: empty cache");
  if (c->n_hi > 0 && (!c->k_hi || !c->v_hi || (c->hi_bits == 8 && (!c->k_hi_meta || !c->v_hi_meta))))
    return fail(MIKV_EINVAL, "decode_attention: null hi-tier buffer");
  if (c->n_lo > 0 && (!c->k_lo || !c->v_lo || !c->k_lo_meta || !c->v_lo_meta))
    return fail(MIKV_EINVAL, "decode_attention: null lo-tier buffer");
  const void* al[] = {c->k_hi, c->v_hi, c->k_hi_meta, c->v_hi_meta, c->k_lo,
                      c->v_lo, c->k_lo_meta, c->v_lo_meta, ws};
  for (const void* p : al)
    if (p && !aligned16(p)) return fail(MIKV_EALIGN, "decode_attention: cache/ws not 16-byte aligned");
  const size_t need = mikv_decode_workspace_bytes(c);
  if (ws_bytes < need) return fail(MIKV_ESHAPE, "decode_attention: workspace %zu < %zu", ws_bytes, need);

  const Plan pl = make_plan(c);
  Params P{};
  P.q = reinterpret_cast<const __half*>(q);
  P.bal = c->balancer;
  P.hi = TierPtrs{static_cast<const uint8_t*>(c->k_hi), static_cast<const uint8_t*>(c->v_hi),
                  static_cast<const uint8_t*>(c->k_hi_meta), static_cast<const uint8_t*>(c->v_hi_meta),
                  c->cap_hi, c->n_hi};
  P.lo = TierPtrs{static_cast<const uint8_t*>(c->k_lo), static_cast<const uint8_t*>(c->v_lo),
                  static_cast<const uint8_t*>(c->k_lo_meta), static_cast<const uint8_t*>(c->v_lo_meta),
                  c->cap_lo, c->n_lo};
  P.Hq = c->Hq;
  P.Hkv = c->Hkv;
  P.rep = c->Hq / c->Hkv;
  P.chunk_hi = pl.chunk_hi;
  P.chunk_lo = pl.chunk_lo;
  P.nsplit_hi = (c->n_hi + pl.chunk_hi - 1) / pl.chunk_hi;
  const int nsplit_lo = (c->n_lo + pl.chunk_lo - 1) / pl.chunk_lo;
  P.smax = pl.smax_hi + pl.smax_lo;
  P.hi_logits = hi_logits;
  const size_t rows = static_cast<size_t>(c->B) * c->Hq * P.smax;
  P.ws_o = static_cast<float*>(ws);
  P.ws_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(rows * kD * sizeof(float), 256));
  const int nsplit = P.nsplit_hi + nsplit_lo;
  dim3 grid(nsplit, c->B * c->Hkv);
  cudaStream_t s = as_stream(stream);
  int e;
  switch (c->hi_bits * 100 + c->lo_bits) {
    case 1602: e = launch_nt<16, 2>(P, grid, s); break;
    case 1604: e = launch_nt<16, 4>(P, grid, s); break;
    case 1608: e = launch_nt<16, 8>(P, grid, s); break;
    case 802: e = launch_nt<8, 2>(P, grid, s); break;
    case 804: e = launch_nt<8, 4>(P, grid, s); break;
    case 808: e = launch_nt<8, 8>(P, grid, s); break;
    default: return fail(MIKV_EUNSUPPORTED, "decode_attention: bits %d/%d", c->hi_bits, c->lo_bits);
  }
  if (e) return e;
  decode_merge_kernel<<<c->B * c->Hq, kD, 0, s>>>(P.ws_o, P.ws_ml, P.smax, nsplit, out, lse);
  return check_launch("decode_merge_kernel");
}
