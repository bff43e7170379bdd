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
//   shared-memory rings filled by 16-byte cp.async (zero-filled past the end),
//   the cache rows marked evict-first in L2 (each is read once per step), so
//   the partials and logits the step's later launches read back stay in L2.
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

#include "quant_device.cuh"

namespace mikv {
int validate_cache_public(const mikv_cache* c, const char* who);

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;        // ring depth per warp (3 CTAs of 4 warps fit per SM)
constexpr float kLogitScale = 0.12751743082459868f;  // log2(e) / sqrt(128)

// Tokens per warp-stage: 16 FP16 rows (8.5 KB with padding), 32 INT8 or INT4 rows, 64 INT2
// rows, so that 4 warps x 2 stages of any format pairing fit 3 CTAs per SM.
__host__ __device__ constexpr int stage_tokens(int bits) { return bits == 16 ? 16 : (bits == 2 ? 64 : 32); }

// CH: keys quantised per channel (groups of 64 slots); a stage then carries its group's key
// meta row (D x (scale, zero), 512 bytes) instead of per-token key meta.
template <int BITS, bool CH = false>
struct Fmt {
  static constexpr bool kQuant = BITS != 16;
  static constexpr int kRB = kD * BITS / 8;                            // bytes per token row
  static constexpr int kRS = kQuant ? kRB : kRB + 16;                  // smem row stride (FP16 padded)
  static constexpr int kST = stage_tokens(BITS);                      // tokens per stage
  static constexpr int kMetaB = kQuant ? 8 : 0;                        // (scale, zero) x 2 groups
  static constexpr int kMetaKB = CH ? kD * 4 : kST * kMetaB;           // key meta bytes per stage
  static constexpr int kOffV = kST * kRS;
  static constexpr int kOffKM = 2 * kST * kRS;
  static constexpr int kOffVM = kOffKM + kMetaKB;
  static constexpr int kStageBytes = 2 * kST * kRS + kMetaKB + kST * kMetaB;
  static constexpr int kCPR = kRB / 16;          // 16-byte chunks per row
  static constexpr int kRowsPerIt = 32 / kCPR;   // rows one warp-wide copy covers
  static constexpr int kGB = 64 * BITS / 8;      // bytes of one 64-channel group
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
  const uint32_t* qf;      // query fragments, [B*Hkv][2][32][kQW]
  uint32_t* qf_out;        // the same buffer, written by the prep kernel
  // per-channel keys: the low tier's closed groups, then the waiting pairs (FP16) as a third
  // tier; qc = the query in the lane order of the low tier's fragments, fp32 [B*Hkv][32][kQC]
  TierPtrs pend;
  int nsplit_lo;
  float* qc;
};
constexpr int kQC = 64;

// ---------------------------------------------------------------------------------
// Shared-memory tiles.  FP16 rows are padded to 272 B, which puts the 8 rows of an
// ldmatrix phase in 8 different 16-byte bank groups.  Code rows (32/64/128 B) keep their
// size and XOR-swizzle their 16-byte chunks with the row bits that repeat the bank
// pattern (every 4 / 2 / 1 rows), so the rows of one fragment load hit different banks.
// The swizzle only depends on row bits below 8, so a thread's fragment offsets are the
// same for every 16-row sub-tile and are computed once.
template <int BITS>
__device__ __forceinline__ int qswz(int r) {
  if constexpr (BITS == 2) return (r >> 2) & 1;
  else if constexpr (BITS == 4) return (r >> 1) & 3;
  else return r & 7;
}
template <int BITS>
__device__ __forceinline__ uint32_t qaddr(int r, int off) {
  return r * Fmt<BITS>::kRS + ((((off >> 4) ^ qswz<BITS>(r))) << 4) + (off & 15);
}

// Per-lane constants of the stage copy: lane l copies the 16-byte chunks l, l+32, ... of
// the stage's contiguous K and V rows; its first chunk lands at smem offset d0 (d1 for odd
// copy iterations of INT8 rows, whose swizzle changes every 4 rows).
template <int BITS>
struct CopyLane {
  uint32_t d0, d1;  // smem offsets of iteration 0 (and odd iterations for INT8)
  int rl;           // row of iteration 0
  __device__ __forceinline__ explicit CopyLane(int lane) {
    using F = Fmt<BITS>;
    const int cc = lane % F::kCPR;
    rl = lane / F::kCPR;
    if constexpr (BITS == 16) {
      d0 = d1 = rl * F::kRS + cc * 16;
    } else {
      d0 = rl * F::kRS + ((cc ^ qswz<BITS>(rl)) << 4);
      d1 = rl * F::kRS + ((cc ^ qswz<BITS>(rl + F::kRowsPerIt)) << 4);
    }
  }
};

// One warp copies a stage: gk/gv point at this lane's first chunk of the stage (stage rows
// are contiguous), gkm/gvm at the stage's first meta row.  FULL: all kST rows valid; else
// rows at or past `nvalid` are zero-filled without being read.
template <int BITS, bool FULL, bool CH = false>
__device__ __forceinline__ void load_stage(uint32_t sb, const uint8_t* gk, const uint8_t* gv,
                                           const uint8_t* gkm, const uint8_t* gvm, int nvalid,
                                           int lane, const CopyLane<BITS>& cl) {
  using F = Fmt<BITS, CH>;
  const uint64_t once = l2_evict_first_policy();  // each cache row is read once per step
#pragma unroll
  for (int it = 0; it < F::kST / F::kRowsPerIt; ++it) {
    const bool ok = FULL || cl.rl + it * F::kRowsPerIt < nvalid;
    const uint32_t dst = ((it & 1) ? cl.d1 : cl.d0) + it * F::kRowsPerIt * F::kRS;
    // a zero-filled chunk reads nothing; it still gets the stage's first chunk (valid)
    cp_async16_once(sb + dst, ok ? gk + it * 512 : gk - lane * 16, ok, once);
    cp_async16_once(sb + F::kOffV + dst, ok ? gv + it * 512 : gv - lane * 16, ok, once);
  }
  if constexpr (F::kQuant) {
    if constexpr (CH) cp_async16(sb + F::kOffKM + lane * 16, gkm + lane * 16, true);  // the group's key meta
#pragma unroll
    for (int it = 0; it < (F::kST + 31) / 32; ++it) {
      const int r = lane + 32 * it;
      if (F::kST % 32 == 0 || r < F::kST) {
        const bool ok = FULL || r < nvalid;
        if constexpr (!CH) cp_async8(sb + F::kOffKM + r * 8, ok ? gkm + r * 8 : gkm, ok);
        cp_async8(sb + F::kOffVM + r * 8, ok ? gvm + r * 8 : gvm, ok);
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// unpacking: codes -> fp16 pairs holding exact integers.
// A code c masked in place at bit 2p (INT2) / 4p (INT4) of a half whose exponent field is
// 0x64 reads as 1024 + c*2^k; one fma.rn.f16x2 by 2^-k with addend -1024*2^-k returns c
// exactly (the true result is a small integer).  Codes above bit 9 are reached with one
// shift of the whole word.  (Feeding the raw bits as fp16 subnormals c*2^k*2^-24 would
// save the fma, but mma.sync on sm_103a did not multiply such operands exactly in our
// measurements: attention errors rose from <1e-4 to ~3e-4.)
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
template <uint32_t MASK>
__device__ __forceinline__ uint32_t mask_magic(uint32_t w) {  // (w & MASK) | 0x64006400, one LOP3
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(w), "n"(MASK), "r"(0x64006400u));
  return d;
}
// (2^-k, -1024*2^-k) f16x2 constants for k = 0, 2, 4, 6, 8
#define MIKV_M4(p) ((p) == 0 ? 0x3C003C00u : (p) == 1 ? 0x34003400u : (p) == 2 ? 0x2C002C00u : (p) == 3 ? 0x24002400u : 0x1C001C00u)
#define MIKV_A4(p) ((p) == 0 ? 0xE400E400u : (p) == 1 ? 0xDC00DC00u : (p) == 2 ? 0xD400D400u : (p) == 3 ? 0xCC00CC00u : 0xC400C400u)
__device__ __forceinline__ void unpack_int2_word_int(uint32_t w, uint32_t (&pr)[8]) {
  pr[0] = hfma2_u32(mask_magic<0x00030003u>(w), MIKV_M4(0), MIKV_A4(0));
  pr[1] = hfma2_u32(mask_magic<0x000C000Cu>(w), MIKV_M4(1), MIKV_A4(1));
  pr[2] = hfma2_u32(mask_magic<0x00300030u>(w), MIKV_M4(2), MIKV_A4(2));
  pr[3] = hfma2_u32(mask_magic<0x00C000C0u>(w), MIKV_M4(3), MIKV_A4(3));
  pr[4] = hfma2_u32(mask_magic<0x03000300u>(w), MIKV_M4(4), MIKV_A4(4));
  const uint32_t w2 = w >> 10;
  pr[5] = hfma2_u32(mask_magic<0x00030003u>(w2), MIKV_M4(0), MIKV_A4(0));
  pr[6] = hfma2_u32(mask_magic<0x000C000Cu>(w2), MIKV_M4(1), MIKV_A4(1));
  pr[7] = hfma2_u32(mask_magic<0x00300030u>(w2), MIKV_M4(2), MIKV_A4(2));
}
__device__ __forceinline__ void unpack_int4_word_int(uint32_t w, uint32_t* pr) {
  pr[0] = hfma2_u32(mask_magic<0x000F000Fu>(w), 0x3C003C00u, 0xE400E400u);
  pr[1] = hfma2_u32(mask_magic<0x00F000F0u>(w), 0x2C002C00u, 0xD400D400u);
  const uint32_t w2 = w >> 8;
  pr[2] = hfma2_u32(mask_magic<0x000F000Fu>(w2), 0x3C003C00u, 0xE400E400u);
  pr[3] = hfma2_u32(mask_magic<0x00F000F0u>(w2), 0x2C002C00u, 0xD400D400u);
}


// K side: the 16 channels [gr*64 + tig*16, +16) of one token row (at smem address
// `addr`) -> 8 pairs; pair p holds local channels (ca(p), cb(p)) in its (low, high) halves.
template <int BITS>
__device__ __forceinline__ void unpack_k16(uint32_t addr, uint32_t (&pr)[8]) {
  if constexpr (BITS == 2) {
    unpack_int2_word_int(lds32(addr), pr);
  } else if constexpr (BITS == 4) {
    const uint2 w = lds64(addr);
    unpack_int4_word_int(w.x, pr);
    unpack_int4_word_int(w.y, pr + 4);
  } else {
    const uint4 w = lds128(addr);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pr[2 * i] = hfma2_u32(__byte_perm(ww[i], 0x64u, 0x4140), 0x3C003C00u, 0xE400E400u);
      pr[2 * i + 1] = hfma2_u32(__byte_perm(ww[i], 0x64u, 0x4342), 0x3C003C00u, 0xE400E400u);
    }
  }
}
// INT4 word pairs: (w & 0xF..) -> codes (0, 4), (w & 0xF0..) -> (1, 5), then after >> 8:
// (2, 6), (3, 7); the second word adds 8.
template <int BITS>
__host__ __device__ constexpr int k_ca(int p) {
  return BITS == 2 ? p : (BITS == 4 ? (p & 3) + (p >> 2) * 8 : 2 * p);
}
template <int BITS>
__host__ __device__ constexpr int k_cb(int p) {
  return BITS == 2 ? p + 8 : (BITS == 4 ? (p & 3) + 4 + (p >> 2) * 8 : 2 * p + 1);
}

// V side: the 8 channels [gr*64 + gid*8, +8) of two consecutive token rows (at smem
// addresses aa, ab) -> 8 pairs, pair c = (code[row a][c], code[row b][c]).
template <int BITS>
__device__ __forceinline__ void unpack_v8(uint32_t aa, uint32_t ab, uint32_t (&pr)[8]) {
  if constexpr (BITS == 2) {
    unpack_int2_word_int(__byte_perm(lds16(aa), lds16(ab), 0x5410), pr);
  } else if constexpr (BITS == 4) {
    const uint32_t ua = lds32(aa), ub = lds32(ab);
    unpack_int4_word_int(__byte_perm(ua, ub, 0x5410), pr);      // channels 0..3
    unpack_int4_word_int(__byte_perm(ua, ub, 0x7632), pr + 4);  // channels 4..7
  } else {
    const uint2 ua = lds64(aa), ub = lds64(ab);
    const uint32_t t0 = __byte_perm(ua.x, ub.x, 0x5140), t1 = __byte_perm(ua.x, ub.x, 0x7362);
    const uint32_t t2 = __byte_perm(ua.y, ub.y, 0x5140), t3 = __byte_perm(ua.y, ub.y, 0x7362);
    const uint32_t m = 0x3C003C00u, a = 0xE400E400u;  // exact integers: (1024 + c) * 1 - 1024
    pr[0] = hfma2_u32(__byte_perm(t0, 0x64u, 0x4140), m, a);
    pr[1] = hfma2_u32(__byte_perm(t0, 0x64u, 0x4342), m, a);
    pr[2] = hfma2_u32(__byte_perm(t1, 0x64u, 0x4140), m, a);
    pr[3] = hfma2_u32(__byte_perm(t1, 0x64u, 0x4342), m, a);
    pr[4] = hfma2_u32(__byte_perm(t2, 0x64u, 0x4140), m, a);
    pr[5] = hfma2_u32(__byte_perm(t2, 0x64u, 0x4342), m, a);
    pr[6] = hfma2_u32(__byte_perm(t3, 0x64u, 0x4140), m, a);
    pr[7] = hfma2_u32(__byte_perm(t3, 0x64u, 0x4342), m, a);
  }
}

// 2^x with one MUFU instruction (ex2.approx.ftz: relative error ~2^-22, exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// (hi, lo) fp16 pair with hi + lo carrying ~21 bits of x: hi = x with its low 13
// mantissa bits cleared (exact in fp16 over the normal range), lo = fp16(x - hi); both
// packed by a single cvt.
__device__ __forceinline__ uint32_t split_pack(float x) {
  const float hi = __uint_as_float(__float_as_uint(x) & 0xffffe000u);
  const __half2 h = __floats2half2_rn(hi, x - hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------------
template <int NT>
struct State {
  float m[NT];          // running max (base-2 logits), uniform over the 8 lanes of a head
  float l[NT];          // per-lane partial denominator
  float zs[NT][2];      // per-lane partial sum_i p_i * zero_v,i per value group
  float o[NT][8][4];    // PV accumulators: 8 channel tiles x (2 rows x (hi, lo))
};

// Per-thread byte offsets of the warp's fragments inside a stage tile (sub-tile 0).
struct FragOffs {
  uint32_t k0, k1;            // codes: K row gid, groups 0/1; FP16: ldmatrix row offset of K
  uint32_t va0, va1, vb0, vb1;  // codes: V rows 2tig / 2tig+1, groups 0/1; FP16: va0 for V^T
};

template <int BITS>
__device__ __forceinline__ FragOffs frag_offsets(int lane) {
  using F = Fmt<BITS>;
  const int gid = lane >> 2, tig = lane & 3;
  FragOffs f{};
  if constexpr (BITS == 16) {
    f.k0 = ((lane & 7) + ((lane >> 3) & 1) * 8) * F::kRS + (lane >> 4) * 16;
    f.va0 = ((lane & 7) + ((lane >> 4) << 3)) * F::kRS + ((lane >> 3) & 1) * 16;
  } else {
    constexpr int TB = 16 * BITS / 8, VB = 8 * BITS / 8;
    f.k0 = qaddr<BITS>(gid, tig * TB);
    f.k1 = qaddr<BITS>(gid, F::kGB + tig * TB);
    f.va0 = qaddr<BITS>(2 * tig, gid * VB);
    f.va1 = qaddr<BITS>(2 * tig, F::kGB + gid * VB);
    f.vb0 = qaddr<BITS>(2 * tig + 1, gid * VB);
    f.vb1 = qaddr<BITS>(2 * tig + 1, F::kGB + gid * VB);
  }
  return f;
}

// One stage of BITS-format tokens for one warp.  The query fragments are pre-scaled by
// log2(e)/sqrt(D), so the accumulators hold base-2 logits.  FULL: all kST rows valid.
// CH: keys quantised per channel; bq then holds this stage's rescaled fragments (q * s per
// channel) and qsum[t][0] the head's zero term sum_c q_c z_c (see rescale_qfrag).
template <int BITS, int NT, bool FULL, bool CH = false>
__device__ __forceinline__ void compute_stage(uint32_t sb, int nvalid, const uint32_t (&bq)[NT][8][2],
                                              const float (&qsum)[NT][2], State<NT>& st,
                                              float* logit_out, int logit_stride, int rep,
                                              int lane, const FragOffs& fo) {
  using F = Fmt<BITS, CH>;
  constexpr int kSub = F::kST / 16;
  constexpr float kLn2 = 0.6931471805599453f;
  const int gid = lane >> 2, tig = lane & 3;
  float x[kSub][NT][2];  // base-2 logits of rows gid, gid+8

  // ---- QK^T for every 16-token sub-tile of the stage
#pragma unroll
  for (int sub = 0; sub < kSub; ++sub) {
    const uint32_t st_k = sb + sub * 16 * F::kRS;
    if constexpr (!F::kQuant) {
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(st_k + fo.k0 + 32 * s, a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma16816(acc[t], a0, a1, a2, a3, bq[t][s][0], bq[t][s][1]);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        x[sub][t][0] = acc[t][0] + acc[t][1];
        x[sub][t][1] = acc[t][2] + acc[t][3];
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
        const uint32_t ka = st_k + (gr ? fo.k1 : fo.k0);
        unpack_k16<BITS>(ka, pa);
        unpack_k16<BITS>(ka + 8 * F::kRS, pb);
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            mma16816(acc[t][gr], pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1],
                     bq[t][gr * 4 + s][0], bq[t][gr * 4 + s][1]);
      }
      if constexpr (CH) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          x[sub][t][0] = ((acc[t][0][0] + acc[t][0][1]) + (acc[t][1][0] + acc[t][1][1])) + qsum[t][0];
          x[sub][t][1] = ((acc[t][0][2] + acc[t][0][3]) + (acc[t][1][2] + acc[t][1][3])) + qsum[t][0];
        }
      } else {
        const uint2 ma = lds64(sb + F::kOffKM + (sub * 16 + gid) * 8);
        const uint2 mb = lds64(sb + F::kOffKM + (sub * 16 + gid + 8) * 8);
        const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&ma.x));
        const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&ma.y));
        const float2 b0 = __half22float2(*reinterpret_cast<const __half2*>(&mb.x));
        const float2 b1 = __half22float2(*reinterpret_cast<const __half2*>(&mb.y));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float da0 = acc[t][0][0] + acc[t][0][1], da1 = acc[t][1][0] + acc[t][1][1];
          const float db0 = acc[t][0][2] + acc[t][0][3], db1 = acc[t][1][2] + acc[t][1][3];
          x[sub][t][0] = a0.x * da0 + a1.x * da1 + a0.y * qsum[t][0] + a1.y * qsum[t][1];
          x[sub][t][1] = b0.x * db0 + b1.x * db1 + b0.y * qsum[t][0] + b1.y * qsum[t][1];
        }
      }
    }
    // natural logits out (important tier) and masking of rows past the end
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int head = t * 4 + tig;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = sub * 16 + gid + 8 * h;
        const bool valid = FULL || r < nvalid;
        if (logit_out != nullptr && head < rep && valid)
          logit_out[head * logit_stride + r] = x[sub][t][h] * kLn2;
        if (!valid) x[sub][t][h] = -INFINITY;
      }
    }
  }

  // ---- online softmax update: one max per stage; the accumulators are rescaled only
  // when some head's running max moved (warp vote)
  float mnew[NT];
  bool moved = false;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float mx = x[0][t][0];
#pragma unroll
    for (int sub = 0; sub < kSub; ++sub) mx = fmaxf(mx, fmaxf(x[sub][t][0], x[sub][t][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mnew[t] = fmaxf(st.m[t], mx);
    moved |= mnew[t] > st.m[t];
  }
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float alpha = fast_exp2(st.m[t] - mnew[t]);  // 0 on the first stage (m = -inf)
      st.m[t] = mnew[t];
      st.l[t] *= alpha;
      st.zs[t][0] *= alpha;
      st.zs[t][1] *= alpha;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[t][j][e] *= alpha;
    }
  }

  // ---- P V for every sub-tile
#pragma unroll
  for (int sub = 0; sub < kSub; ++sub) {
    const uint32_t st_v = sb + F::kOffV + sub * 16 * F::kRS;
    float p[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      p[t][0] = fast_exp2(x[sub][t][0] - mnew[t]);
      p[t][1] = fast_exp2(x[sub][t][1] - mnew[t]);
      st.l[t] += p[t][0] + p[t][1];
    }
    if constexpr (!F::kQuant) {
      uint32_t bp[NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) bp[t][h] = movmatrix_t(split_pack(p[t][h]));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(st_v + fo.va0 + 32 * j, a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma16816(st.o[t][j], a0, a1, a2, a3, bp[t][0], bp[t][1]);
      }
    } else {
      // value scale/zero of rows gid, gid+8 for both groups
      const uint2 ma = lds64(sb + F::kOffVM + (sub * 16 + gid) * 8);
      const uint2 mb = lds64(sb + F::kOffVM + (sub * 16 + gid + 8) * 8);
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
          bp[t][gr][0] = movmatrix_t(split_pack(p[t][0] * va[gr].x));
          bp[t][gr][1] = movmatrix_t(split_pack(p[t][1] * vb[gr].x));
        }
      }
#pragma unroll
      for (int gr = 0; gr < 2; ++gr) {
        uint32_t v01[8], v89[8];
        const uint32_t aa = st_v + (gr ? fo.va1 : fo.va0), ab = st_v + (gr ? fo.vb1 : fo.vb0);
        unpack_v8<BITS>(aa, ab, v01);
        unpack_v8<BITS>(aa + 8 * F::kRS, ab + 8 * F::kRS, v89);
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

// Query fragments in the lane order of the partial kernel: word 16t + 2s + i of a lane is
// bq[t][s][i], words 32..35 qsum[NT][2]; [units][2 formats][32 lanes][kQW].
constexpr int kQW = 36;

template <int NT>
__device__ __forceinline__ void load_qfrag(const uint32_t* qf, int unit, int tier, int lane,
                                           uint32_t (&bq)[NT][8][2], float (&qsum)[NT][2]) {
  const uint4* src =
      reinterpret_cast<const uint4*>(qf + ((static_cast<long>(unit) * 2 + tier) * 32 + lane) * kQW);
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint4 w = src[t * 4 + q4];
      bq[t][2 * q4][0] = w.x;
      bq[t][2 * q4][1] = w.y;
      bq[t][2 * q4 + 1][0] = w.z;
      bq[t][2 * q4 + 1][1] = w.w;
    }
  const uint4 s = src[8];
  qsum[0][0] = __uint_as_float(s.x);
  qsum[0][1] = __uint_as_float(s.y);
  if constexpr (NT == 2) {
    qsum[1][0] = __uint_as_float(s.z);
    qsum[1][1] = __uint_as_float(s.w);
  }
}

// Query fragments of one (batch, key head) for both tier formats, by one CTA of >= 256
// threads.  Thread (f, c) of the first 256 stages channel c of every query head of the group
// for format f (0 = important tier, 1 = low tier): pre-scaled by log2(e)/sqrt(D) and, for a
// quantised format, divided by the balancer, as an fp16 (hi, lo) pair; with the 64-channel
// group sums of the same scaled values.  Warp 0 (format 0) and warp 4 (format 1) then gather
// their lane-order fragments (word 16t + 2s + i = bq[t][s][i], words 32..35 = qsum[NT][2]).
// Every thread of the CTA must call this (it holds a barrier).
template <int HI, int LO, int NT, bool CK = false>
__device__ __forceinline__ void prep_unit(const Params& P, int unit) {
  __shared__ uint32_t sq[2][8][kD];   // (hi, lo) pairs
  __shared__ float sgs[2][8][4];      // per-warp partial sums: [format][head][warp of the format]
  __shared__ float sqf[CK ? 8 : 1][kD];  // per-channel keys: the scaled query in fp32
  const int t = threadIdx.x, lane = t & 31;
  const int b = unit / P.Hkv, g = unit % P.Hkv;
  if (t < 256) {
    const int f = t >> 7, c = t & (kD - 1);
    const bool quant = f == 0 ? Fmt<HI>::kQuant : Fmt<LO>::kQuant;
    const float bb = (quant && P.bal) ? P.bal[static_cast<long>(unit) * kD + c] : 1.f;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float x = 0.f;
      if (h < P.rep) {
        x = __half2float(P.q[(static_cast<long>(b) * P.Hq + g * P.rep + h) * kD + c]);
        if (quant && P.bal) x = __fdiv_rn(x, bb);
        x *= kLogitScale;
      }
      sq[f][h][c] = split_pack(x);
      if (CK && f == 1) sqf[h][c] = x;
      float sum = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) sgs[f][h][c >> 5] = sum;
    }
  }
  __syncthreads();
  if (t < 256 && (t & 127) < 32) {
    const int f = t >> 7;
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t w[kQW];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
      const int head = tt * 4 + (gid >> 1);
      const int shift = (gid & 1) * 16;  // hi part in column 2h, lo part in column 2h + 1
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        int c0, c1, c2, c3;
        if ((f == 0 ? HI : LO) == 16) {
          c0 = s2 * 16 + 2 * tig;
          c1 = c0 + 1;
          c2 = c0 + 8;
          c3 = c0 + 9;
        } else {
          const int bits = f == 0 ? HI : LO;
          const int gr = s2 >> 2, sp = s2 & 3, base = gr * 64 + tig * 16;
          c0 = base + (bits == 2 ? k_ca<2>(2 * sp) : bits == 4 ? k_ca<4>(2 * sp) : k_ca<8>(2 * sp));
          c1 = base + (bits == 2 ? k_cb<2>(2 * sp) : bits == 4 ? k_cb<4>(2 * sp) : k_cb<8>(2 * sp));
          c2 = base + (bits == 2 ? k_ca<2>(2 * sp + 1) : bits == 4 ? k_ca<4>(2 * sp + 1) : k_ca<8>(2 * sp + 1));
          c3 = base + (bits == 2 ? k_cb<2>(2 * sp + 1) : bits == 4 ? k_cb<4>(2 * sp + 1) : k_cb<8>(2 * sp + 1));
        }
        const uint32_t* row = sq[f][head];
        w[tt * 16 + 2 * s2] = ((row[c0] >> shift) & 0xffffu) | (((row[c1] >> shift) & 0xffffu) << 16);
        w[tt * 16 + 2 * s2 + 1] = ((row[c2] >> shift) & 0xffffu) | (((row[c3] >> shift) & 0xffffu) << 16);
      }
    }
#pragma unroll
    for (int i = 16 * NT; i < 32; ++i) w[i] = 0u;
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const int head = tt * 4 + tig;
      const bool on = tt < NT;
      w[32 + 2 * tt] = __float_as_uint(on ? sgs[f][head][0] + sgs[f][head][1] : 0.f);
      w[33 + 2 * tt] = __float_as_uint(on ? sgs[f][head][2] + sgs[f][head][3] : 0.f);
    }
    uint4* dst = reinterpret_cast<uint4*>(P.qf_out + ((static_cast<long>(unit) * 2 + f) * 32 + lane) * kQW);
#pragma unroll
    for (int i = 0; i < kQW / 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    if (CK && f == 1) {  // the same lane order, fp32, for the per-stage rescaling
      float* qd = P.qc + (static_cast<long>(unit) * 32 + lane) * kQC;
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int head = tt * 4 + (gid >> 1);
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          const int sp = s2 & 3, base = (s2 >> 2) * 64 + tig * 16;
          const int c0 = base + k_ca<LO>(2 * sp), c1 = base + k_cb<LO>(2 * sp);
          const int c2 = base + k_ca<LO>(2 * sp + 1), c3 = base + k_cb<LO>(2 * sp + 1);
          const bool on = tt < NT;
          reinterpret_cast<float4*>(qd + tt * 32 + s2 * 4)[0] =
              on ? make_float4(sqf[head][c0], sqf[head][c1], sqf[head][c2], sqf[head][c3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

// The query fragments of every (batch, key head): one CTA of 256 threads per unit.
template <int HI, int LO, int NT, bool CK>
__global__ void __launch_bounds__(256) decode_qprep_kernel(Params P) {
  pdl_wait();
  pdl_trigger();
  prep_unit<HI, LO, NT, CK>(P, blockIdx.x);
}

// First kernel of a decode step, one CTA of 288 threads per (batch, key head): the last warp
// appends the new token to the important tier (and clears the unit's demotion ticket), the
// rest prepare the query fragments.
template <int HI, int LO, int NT, bool CK>
__global__ void __launch_bounds__(288) decode_step_prep_kernel(AppendArgs a, Params P) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x >= 256) append_item(a, blockIdx.x, threadIdx.x & 31);
  prep_unit<HI, LO, NT, CK>(P, blockIdx.x);
}

// Per-channel keys: the query fragments of one stage.  The stage's keys carry a scale s_c and
// zero z_c per channel (the group's meta row in shared memory at `km`), so
//   q . k~ = sum_c (q_c s_c) code_c + sum_c q_c z_c.
// Each lane forms its fragment words from the fp32 query (already scaled by log2(e)/sqrt(D),
// in its own lane order, `q32`): q_c s_c split into fp16 (hi, lo) parts as the prep does, the
// part of its column (hi for even gid, lo for odd); and the zero term of its head, summed over
// the 4 lanes that hold the head's 128 channels, then handed to the lanes whose accumulator
// rows belong to that head (zt[t] for head t * 4 + tig).
__device__ __forceinline__ uint32_t part_pack(float a, float b, bool lo_part) {
  const float ha = __uint_as_float(__float_as_uint(a) & 0xffffe000u);
  const float hb = __uint_as_float(__float_as_uint(b) & 0xffffe000u);
  const __half2 h = __floats2half2_rn(lo_part ? a - ha : ha, lo_part ? b - hb : hb);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BITS, int NT>
__device__ __forceinline__ void rescale_qfrag(uint32_t km, const float* q32, int lane, uint32_t (&bqs)[NT][8][2],
                                              float (&zt)[NT][2]) {
  const int gid = lane >> 2, tig = lane & 3;
  const bool lo_part = (gid & 1) != 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float zp = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) {
      const float4 qv = __ldg(reinterpret_cast<const float4*>(q32 + t * 32 + s2 * 4));
      const int sp = s2 & 3, base = (s2 >> 2) * 64 + tig * 16;
      const int c0 = base + k_ca<BITS>(2 * sp), c1 = base + k_cb<BITS>(2 * sp);
      const int c2 = base + k_ca<BITS>(2 * sp + 1), c3 = base + k_cb<BITS>(2 * sp + 1);
      uint32_t w0 = lds32(km + c0 * 4), w1 = lds32(km + c1 * 4), w2 = lds32(km + c2 * 4), w3 = lds32(km + c3 * 4);
      const float2 m0 = __half22float2(*reinterpret_cast<const __half2*>(&w0));
      const float2 m1 = __half22float2(*reinterpret_cast<const __half2*>(&w1));
      const float2 m2 = __half22float2(*reinterpret_cast<const __half2*>(&w2));
      const float2 m3 = __half22float2(*reinterpret_cast<const __half2*>(&w3));
      zp = fmaf(qv.x, m0.y, fmaf(qv.y, m1.y, fmaf(qv.z, m2.y, fmaf(qv.w, m3.y, zp))));
      bqs[t][s2][0] = part_pack(qv.x * m0.x, qv.y * m1.x, lo_part);
      bqs[t][s2][1] = part_pack(qv.z * m2.x, qv.w * m3.x, lo_part);
    }
    zp += __shfl_xor_sync(0xffffffffu, zp, 1);
    zp += __shfl_xor_sync(0xffffffffu, zp, 2);
    zt[t][0] = __shfl_sync(0xffffffffu, zp, 8 * tig);
    zt[t][1] = 0.f;
  }
}

// One CTA's chunk of one tier.  fmt: which query fragments (0: the important tier's format,
// 1: the low tier's); logits: write the natural logits of its tokens (important tier);
// split_index: the CTA's row in the split workspace.  CH: per-channel keys (the low tier).
template <int BITS, int NT, bool CH = false>
__device__ void run_tier(const Params& P, const TierPtrs& tier, int unit, int split, int chunk,
                         int fmt, bool logits, int split_index, uint8_t* smem) {
  using F = Fmt<BITS, CH>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = unit / P.Hkv, g = unit % P.Hkv;
  const int rep = P.rep;

  const int t_begin = split * chunk;
  const int t_end = min(tier.n, t_begin + chunk);
  const int nst = (t_end - t_begin + F::kST - 1) / F::kST;   // stages in this CTA
  const int my_st = nst > warp ? (nst - warp + kWarps - 1) / kWarps : 0;  // this warp's share
  uint8_t* ring = smem + warp * (kStages * F::kStageBytes);  // this warp's ring
  const uint32_t ring_s = smem_u32(ring);
  // warp w handles stages w, w+4, ...; stage pointers advance by a constant stride
  const long row0 = static_cast<long>(unit) * tier.cap + t_begin + warp * F::kST;
  constexpr long kRowStride = static_cast<long>(kWarps) * F::kST;
  const CopyLane<BITS> cl(lane);
  const uint8_t* gk = tier.k + row0 * F::kRB + lane * 16;
  const uint8_t* gv = tier.v + row0 * F::kRB + lane * 16;
  const uint8_t* gkm = F::kQuant ? tier.km + (CH ? 0 : row0 * 8) : nullptr;
  const uint8_t* gvm = F::kQuant ? tier.vm + row0 * 8 : nullptr;
  int tok_issue = t_begin + warp * F::kST;  // first token of the next stage to issue
  int issued = 0;
  auto issue = [&]() {
    if (issued < my_st) {
      const uint32_t sb = ring_s + (issued % kStages) * F::kStageBytes;
      const int nv = t_end - tok_issue;
      // per-channel keys: the meta row of the stage's group of 64 slots
      const uint8_t* km = CH ? gkm + (static_cast<long>(unit) * (tier.cap / kGS) + tok_issue / kGS) * (kD * 4) : gkm;
      if (nv >= F::kST) load_stage<BITS, true, CH>(sb, gk, gv, km, gvm, nv, lane, cl);
      else load_stage<BITS, false, CH>(sb, gk, gv, km, gvm, nv, lane, cl);
      gk += kRowStride * F::kRB;
      gv += kRowStride * F::kRB;
      if constexpr (F::kQuant) {
        if constexpr (!CH) gkm += kRowStride * 8;
        gvm += kRowStride * 8;
      }
      tok_issue += kRowStride;
    }
    ++issued;
    cp_async_commit();
  };
  issue();  // first stage in flight while the query fragments load

  // this tier's query fragments, prepared once per (batch, key head) by the prep kernel
  uint32_t bq[NT][8][2];
  float qsum[NT][2];
  if constexpr (!CH) load_qfrag<NT>(P.qf, unit, fmt, lane, bq, qsum);
  const float* q32 = CH ? P.qc + (static_cast<long>(unit) * 32 + lane) * kQC : nullptr;

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

  float* lrow = nullptr;
  if (logits && P.hi_logits)
    lrow = P.hi_logits + (static_cast<long>(b) * P.Hq + g * rep) * tier.cap;

  const FragOffs fo = frag_offsets<BITS>(lane);
  for (int i = 1; i < kStages - 1; ++i) issue();  // ring prologue (stage 0 is already issued)
  int tok0 = t_begin + warp * F::kST;
  for (int k = 0; k < my_st; ++k) {
    issue();  // stage k + kStages - 1 (or an empty group)
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int nv = min(F::kST, t_end - tok0);
    const uint32_t sb = ring_s + (k % kStages) * F::kStageBytes;
    float* lo = lrow ? lrow + tok0 : nullptr;
    if constexpr (CH) rescale_qfrag<BITS, NT>(sb + F::kOffKM, q32, lane, bq, qsum);
    if (nv == F::kST) compute_stage<BITS, NT, true, CH>(sb, nv, bq, qsum, st, lo, tier.cap, rep, lane, fo);
    else compute_stage<BITS, NT, false, CH>(sb, nv, bq, qsum, st, lo, tier.cap, rep, lane, fo);
    __syncwarp();
    tok0 += kRowStride;
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

// Splits [0, nsplit_hi): the important tier; then the low tier; with per-channel keys (CK)
// the low tier's closed groups, then one CTA over the waiting pairs (FP16, attended with the
// important tier's query fragments, no logits).  Three CTAs per SM; the two-column-tile form
// (NT = 2, five to eight query heads per key head) takes two, with the registers to hold its
// doubled fragments and accumulators without spills (measured at five heads per key head,
// batch 1: 27.1 -> 25.3 us per attention launch).
template <int HI, int LO, int NT, bool CK>
__global__ void __launch_bounds__(kThreads, NT == 2 ? 2 : 3) decode_partial_kernel(Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const int unit = blockIdx.y;
  const int sx = blockIdx.x;
  if (sx < P.nsplit_hi) run_tier<HI, NT>(P, P.hi, unit, sx, P.chunk_hi, 0, true, sx, smem);
  else if (!CK || sx < P.nsplit_hi + P.nsplit_lo)
    run_tier<LO, NT, CK>(P, P.lo, unit, sx - P.nsplit_hi, P.chunk_lo, 1, false, sx, smem);
  else if constexpr (CK) run_tier<16, NT>(P, P.pend, unit, 0, kGS, 0, false, sx, smem);
}

// K8: merge the split partials (base-2 max m, sum l, unnormalised o) of one query head
// (row = b*Hq + h) into its output row and natural log-sum-exp.  G groups of threads fold the
// splits: group g takes splits g, g+G, g+2G, ... in ascending order, and the group sums are
// then added in group order.  G is the smallest power of two that leaves at most 8 splits to a
// group (at most 32); a CTA holds G groups of kD / chunks channels (thread = channel), so a
// row spreads over `chunks` CTAs once G passes 8.  G depends on nsplit only, so every caller
// of this kernel gets the same bits.
__host__ __device__ inline int merge_groups(int nsplit) {
  int g = 1;
  while (g < 32 && g * 8 < nsplit) g *= 2;
  return g;
}
__host__ __device__ inline int merge_chunks(int nsplit) { return merge_groups(nsplit) > 8 ? merge_groups(nsplit) / 8 : 1; }

__global__ void __launch_bounds__(1024) decode_merge_kernel(const float* __restrict__ ws_o,
                                                            const float* __restrict__ ws_ml,
                                                            int smax, int nsplit,
                                                            float* __restrict__ out,
                                                            float* __restrict__ lse) {
  __shared__ float so[1024];  // (group - 1, channel) sums of groups 1 .. G-1
  __shared__ float sl[32];
  __shared__ float smx[32];
  pdl_wait();
  pdl_trigger();
  const int chunks = merge_chunks(nsplit);
  const int G = blockDim.x * chunks / kD, CC = blockDim.x / G;
  const int cl = threadIdx.x % CC, gi = threadIdx.x / CC;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long row = blockIdx.x / chunks;
  const int c = static_cast<int>(blockIdx.x % chunks) * CC + cl;
  const float* ml = ws_ml + row * smax * 2;
  // the running maxima: max is exact in any order
  float M = -INFINITY;
  for (int s = threadIdx.x; s < nsplit; s += blockDim.x) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) smx[warp] = M;
  __syncthreads();
  M = smx[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) M = fmaxf(M, smx[w]);
  float L = 0.f, O = 0.f;
#pragma unroll 8
  for (int s = gi; s < nsplit; s += G) {
    const float ms = ml[2 * s];
    const float sc = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
    L += sc * ml[2 * s + 1];
    O += sc * ws_o[(row * smax + s) * kD + c];
  }
  if (gi > 0) {
    so[(gi - 1) * CC + cl] = O;
    if (cl == 0) sl[gi - 1] = L;
  }
  __syncthreads();
  if (gi > 0) return;
  for (int g = 1; g < G; ++g) {
    O += so[(g - 1) * CC + cl];
    L += sl[g - 1];
  }
  out[row * kD + c] = O / L;
  if (c == 0) lse[row] = (M + log2f(L)) * 0.69314718055994531f;
}

// End of a decode step after the merge, grid (B*Hkv units, chunks of kEpiChunk slots): add
// this step's attention to the H2O score of every important slot (the arithmetic of the
// separate decode score update) and, when the important tier is over budget, demote the
// victim: the slot with the lowest score, latest position first among equal scores, among
// positions < limit (as the separate demotion select + append).  Each CTA reduces its
// chunk's candidate, publishes it, and takes a ticket; the CTA that takes the unit's last
// ticket reduces the published candidates and moves the victim.  No CTA waits on another.
// The tickets are cleared by the step's append.
constexpr int kEpiThreads = 256;
constexpr int kEpiPer = 4;
constexpr int kEpiChunk = kEpiThreads * kEpiPer;

struct EpiArgs {
  const float* logits;  // [B][Hq][cap_hi]
  const float* lse;     // [B][Hq], from the merge
  int Hq, Hkv, nchunk;
  int demote, limit;
  DemoteArgs da;        // counts after this step's append
  float* cand_s;        // [B*Hkv][nchunk] per-chunk candidates
  int* cand_p;
  int* cand_j;
  unsigned* ticket;     // [B*Hkv]
};

// (s1, p1, j1) is a better victim than (s0, p0, j0); j < 0 marks "no candidate"
__device__ __forceinline__ bool victim_better(float s1, int p1, int j1, float s0, int p0, int j0) {
  return j1 >= 0 && (j0 < 0 || s1 < s0 || (s1 == s0 && p1 > p0));
}

__device__ __forceinline__ void victim_warp_min(float& s, int& p, int& j) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int p2 = __shfl_xor_sync(0xffffffffu, p, o);
    const int j2 = __shfl_xor_sync(0xffffffffu, j, o);
    if (victim_better(s2, p2, j2, s, p, j)) {
      s = s2;
      p = p2;
      j = j2;
    }
  }
}

template <int REP>
__global__ void __launch_bounds__(kEpiThreads) decode_score_demote_kernel(EpiArgs a) {
  __shared__ float s_lse[REP];
  __shared__ float ws_s[kEpiThreads / 32];
  __shared__ int ws_p[kEpiThreads / 32], ws_j[kEpiThreads / 32];
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const long unit = blockIdx.x;
  const int chunk = blockIdx.y;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int b = static_cast<int>(unit / a.Hkv), g = static_cast<int>(unit % a.Hkv);
  const long row0 = static_cast<long>(b) * a.Hq + static_cast<long>(g) * REP;
  const int cap = a.da.cap_hi, n = a.da.n_hi;
  const long ubase = unit * cap;
  // every load of the thread's slots is issued before the first use
  float lg[kEpiPer][REP], sc[kEpiPer];
  int ps[kEpiPer];
#pragma unroll
  for (int i = 0; i < kEpiPer; ++i) {
    const int j = chunk * kEpiChunk + i * kEpiThreads + t;
    const bool in = j < n;
#pragma unroll
    for (int r = 0; r < REP; ++r) lg[i][r] = in ? a.logits[(row0 + r) * cap + j] : 0.f;
    sc[i] = in ? a.da.scores[ubase + j] : 0.f;
    ps[i] = (in && a.demote) ? a.da.pos_hi[ubase + j] : 0;
  }
  if (t < REP) s_lse[t] = a.lse[row0 + t];
  __syncthreads();
  float bs = INFINITY;
  int bp = -1, bj = -1;
#pragma unroll
  for (int i = 0; i < kEpiPer; ++i) {
    const int j = chunk * kEpiChunk + i * kEpiThreads + t;
    if (j < n) {
      float add = 0.f;
#pragma unroll
      for (int r = 0; r < REP; ++r) add += expf(lg[i][r] - s_lse[r]);
      const float sv = sc[i] + add;
      a.da.scores[ubase + j] = sv;
      const int p = ps[i];
      if (a.demote && p < a.limit && victim_better(sv, p, j, bs, bp, bj)) {
        bs = sv;
        bp = p;
        bj = j;
      }
    }
  }
  if (!a.demote) return;
  victim_warp_min(bs, bp, bj);
  if (lane == 0) {
    ws_s[warp] = bs;
    ws_p[warp] = bp;
    ws_j[warp] = bj;
  }
  __syncthreads();
  if (t == 0) {
    for (int w = 1; w < kEpiThreads / 32; ++w)
      if (victim_better(ws_s[w], ws_p[w], ws_j[w], bs, bp, bj)) {
        bs = ws_s[w];
        bp = ws_p[w];
        bj = ws_j[w];
      }
    const long ci = unit * a.nchunk + chunk;
    a.cand_s[ci] = bs;
    a.cand_p[ci] = bp;
    a.cand_j[ci] = bj;
    __threadfence();  // scores and candidate visible before the ticket is taken
    s_last = atomicAdd(&a.ticket[unit], 1u) == static_cast<unsigned>(a.nchunk - 1);
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();  // every other chunk's scores and candidate are visible from here on
  bs = INFINITY;
  bp = bj = -1;
  for (int k = lane; k < a.nchunk; k += 32) {
    const long ci = unit * a.nchunk + k;
    const float s2 = __ldcg(a.cand_s + ci);
    const int p2 = __ldcg(a.cand_p + ci), j2 = __ldcg(a.cand_j + ci);
    if (victim_better(s2, p2, j2, bs, bp, bj)) {
      bs = s2;
      bp = p2;
      bj = j2;
    }
  }
  victim_warp_min(bs, bp, bj);
  demote_one(a.da, unit, bj, lane);
}

// ---------------------------------------------------------------------------------
// host-side split plan
int row_cost(int bits) { return bits == 16 ? 512 : 2 * (kD * bits / 8) + 16; }
// Relative time per byte of a tier: low-bit codes cost more unpacking per byte.  INT2 at 3.0
// and INT4 at 2.0, above their plain rate ratios, because in a mixed launch smaller low-bit
// chunks balance the grid better (measured over INT2 2.0 .. 4.0 and INT4 1.5 .. 2.5: FP16 /
// INT2 at 20 % 124.1 -> 120.2 us, Llama-2-7B 43.4 -> 41.6 us, FP16 / INT4 at 10 % 132.9 ->
// 129.8 us, INT4 / INT2 111.3 -> 108.6 us; INT2 only 106.0 -> 107.1 us).
double byte_weight(int bits) { return bits == 16 ? 1.0 : bits == 8 ? 1.25 : bits == 4 ? 2.0 : 3.0; }
// Makespan model of the split-K grid, fitted to measured attention times over several
// plans and cache shapes: a CTA costs its weighted bytes plus a fixed kCtaOverhead, the
// resident slots share the total, and the tail adds kTailFactor times the largest CTA.
constexpr double kCtaOverhead = 183.0 * 1024;
constexpr double kTailFactor = 2.13;
#ifndef MIKV_MIN_WAVES
#define MIKV_MIN_WAVES 2.5
#endif
constexpr double kMinWaves = MIKV_MIN_WAVES;  // keep at least this many waves when the cache allows
// With few (batch, key head) units every unit is cut into very many splits to fill that many
// waves, and the per-CTA fixed cost and the merge of the splits dominate: below this many
// units one wave suffices (measured at batch 1 / 8 key heads: 37.9 vs 39.5 us per layer-step;
// at 256 units fewer waves were slower).
constexpr int kFewUnits = 64;
// CTA slots per SM that the plan counts: three (the two-column-tile form runs two per SM; its
// plans were measured with this count).
constexpr int kCtasPerSm = 3;

struct Plan {
  int chunk_hi, chunk_lo, smax_hi, smax_lo;
};

// Split plan from the capacities (so the workspace fits every count up to them).  Each tier
// is cut into equal chunks of whole warp-stages; over a geometric range of per-CTA targets
// the plan with the lowest modelled makespan (among those with >= kMinWaves waves, one wave
// below kFewUnits units) wins.
Plan make_plan(const mikv_cache* c) {
  const double units = static_cast<double>(c->B) * c->Hkv;
  const double slots = static_cast<double>(kNumSMs) * kCtasPerSm;
  const double wb_hi = row_cost(c->hi_bits) * byte_weight(c->hi_bits);  // per token
  // five to eight query heads per key head double the low tier's MMA and softmax work per
  // byte (the two-column-tile form): its bytes weigh 1.5 times more (measured at the
  // Qwen2.5-32B shape: 25.4 -> 25.0 us per attention launch, 37.7 -> 36.3 us per step; 2.0 was
  // slower than 1.0)
  const double wb_lo = row_cost(c->lo_bits) * byte_weight(c->lo_bits) * (c->Hq / c->Hkv > 4 ? 1.5 : 1.0);
  const double total = units * (c->cap_hi * wb_hi + c->cap_lo * wb_lo);
  auto chunk_for = [](int cap, double wb, int bits, double target) {
    const int quantum = kWarps * stage_tokens(bits);
    const int ns = std::max(1, static_cast<int>(cap * wb / target + 0.5));
    const int chunk = (std::max(cap, 1) + ns - 1) / ns;
    return std::max(quantum, (chunk + quantum - 1) / quantum * quantum);
  };
  Plan best{}, first{};
  double best_t = INFINITY;
  bool have_first = false;
  for (double target = 32.0 * 1024; target <= 2048.0 * 1024; target *= 1.125) {
    Plan p;
    p.chunk_hi = chunk_for(c->cap_hi, wb_hi, c->hi_bits, target);
    p.chunk_lo = chunk_for(c->cap_lo, wb_lo, c->lo_bits, target);
    p.smax_hi = (c->cap_hi + p.chunk_hi - 1) / p.chunk_hi;
    p.smax_lo = (c->cap_lo + p.chunk_lo - 1) / p.chunk_lo;
    if (!have_first) {
      first = p;
      have_first = true;
    }
    const double ctas = units * (p.smax_hi + p.smax_lo);
    if (ctas < (units < kFewUnits ? 1.0 : kMinWaves) * slots) continue;
    const double largest = std::max(std::min(p.chunk_hi, c->cap_hi) * wb_hi,
                                    std::min(p.chunk_lo, c->cap_lo) * wb_lo);
    const double t = (total + ctas * kCtaOverhead) / slots + kTailFactor * largest;
    if (t < best_t) {
      best_t = t;
      best = p;
    }
  }
  return best_t < INFINITY ? best : first;
}

thread_local cudaEvent_t t_ev_begin = nullptr, t_ev_end = nullptr;

int record_hook(cudaEvent_t ev, cudaStream_t s) {
  if (ev == nullptr) return MIKV_OK;
  const cudaError_t err = cudaEventRecord(ev, s);
  if (err == cudaSuccess) return MIKV_OK;
  (void)cudaGetLastError();
  return fail(MIKV_ECUDA, "attention event record: %s", cudaGetErrorString(err));
}

// The query-fragment prep, then the split-K partial kernel (PDL after the prep); `after`:
// the kernel launched just before on `s` is one of ours, so the prep may overlap its tail.
template <int HI, int LO, int NT, bool CK>
int launch(const Params& P, dim3 grid, cudaStream_t s, bool after, const AppendArgs* step) {
  const dim3 pgrid(grid.y);
  if (step != nullptr) {  // the step's token append and the query prep in one launch
    if (int e = check_launch_after(launch_after(decode_step_prep_kernel<HI, LO, NT, CK>, pgrid, dim3(288),
                                                0, s, *step, P),
                                   "decode_step_prep_kernel"))
      return e;
  } else if (after) {
    auto prep = decode_qprep_kernel<HI, LO, NT, CK>;
    const dim3 pblock(256);
    if (int e = check_launch_after(launch_after(prep, pgrid, pblock, 0, s, P), "decode_qprep_kernel"))
      return e;
  } else {
    decode_qprep_kernel<HI, LO, NT, CK><<<pgrid, 256, 0, s>>>(P);
    if (int e = check_launch("decode_qprep_kernel")) return e;
  }
  const int smem = kWarps * kStages * std::max(Fmt<HI>::kStageBytes, Fmt<LO, CK>::kStageBytes);
  auto kern = decode_partial_kernel<HI, LO, NT, CK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("decode_partial_kernel attribute");
  if (int e = record_hook(t_ev_begin, s)) return e;
  if (int e = check_launch_after(launch_after(kern, grid, dim3(kThreads), smem, s, P),
                                 "decode_partial_kernel"))
    return e;
  return record_hook(t_ev_end, s);
}

template <int HI, int LO, bool CK = false>
int launch_nt(const Params& P, dim3 grid, cudaStream_t s, bool after, const AppendArgs* step) {
  return P.rep <= 4 ? launch<HI, LO, 1, CK>(P, grid, s, after, step)
                    : launch<HI, LO, 2, CK>(P, grid, s, after, step);
}

}  // namespace
}  // namespace mikv

using namespace mikv;

namespace mikv {
namespace {
// Decode workspace: split partials (o, then (m, l)), query fragments, and with per-channel
// keys the fp32 query in the low tier's lane order; one more split row for the waiting pairs.
struct DecWs {
  size_t o, ml, qf, qc, total;
  int smax;
};
DecWs dec_ws_layout(const mikv_cache* c) {
  const Plan p = make_plan(c);
  const bool ck = c->key_mode == MIKV_KEYS_PER_CHANNEL;
  DecWs w;
  w.smax = p.smax_hi + p.smax_lo + (ck ? 1 : 0);
  const size_t rows = static_cast<size_t>(c->B) * c->Hq * w.smax;
  const size_t units = static_cast<size_t>(c->B) * c->Hkv;
  w.o = 0;
  w.ml = align_up(rows * kD * sizeof(float), 256);
  w.qf = w.ml + align_up(rows * 2 * sizeof(float), 256);
  w.qc = w.qf + align_up(units * 2 * 32 * kQW * sizeof(uint32_t), 256);
  w.total = w.qc + (ck ? align_up(units * 32 * kQC * sizeof(float), 256) : 0);
  return w;
}
}  // namespace
}  // namespace mikv

extern "C" size_t mikv_decode_workspace_bytes(const mikv_cache* c) {
  if (validate_cache_public(c, "decode_workspace_bytes") != MIKV_OK) return 0;
  return dec_ws_layout(c).total;
}

namespace mikv {
int append_args(bool hi, const uint16_t* k, const uint16_t* v, int src_len, const int32_t* src_pos,
                int n_tokens, int pos_base, const float* src_scores, const mikv_cache* c,
                unsigned* ticket, AppendArgs& a);
int demote_args(const mikv_cache* c, const int32_t* victim, DemoteArgs& a);
int channel_close_waiting(const mikv_cache* c, cudaStream_t s);

namespace {
// Validate the cache for attention and fill the partial-kernel parameters.
int prepare_decode(const uint16_t* q, const mikv_cache* c, float* hi_logits, void* ws,
                   size_t ws_bytes, Params& P, int& nsplit, const char* who) {
  if (c->n_hi + c->n_lo < 1) return fail(MIKV_ESHAPE, "%s: empty cache", who);
  if (c->n_hi > 0 && (!c->k_hi || !c->v_hi || (c->hi_bits != 16 && (!c->k_hi_meta || !c->v_hi_meta))))
    return fail(MIKV_EINVAL, "%s: null hi-tier buffer", who);
  if (c->n_lo > 0 && (!c->k_lo || !c->v_lo || !c->k_lo_meta || !c->v_lo_meta))
    return fail(MIKV_EINVAL, "%s: null lo-tier buffer", who);
  const void* al[] = {c->k_hi, c->v_hi, c->k_hi_meta, c->v_hi_meta, c->k_lo,
                      c->v_lo, c->k_lo_meta, c->v_lo_meta, ws};
  for (const void* p : al)
    if (p && !aligned16(p)) return fail(MIKV_EALIGN, "%s: cache/ws not 16-byte aligned", who);
  const size_t need = mikv_decode_workspace_bytes(c);
  if (ws_bytes < need) return fail(MIKV_ESHAPE, "%s: workspace %zu < %zu", who, ws_bytes, need);
  const Plan pl = make_plan(c);
  const bool ck = c->key_mode == MIKV_KEYS_PER_CHANNEL;
  P = Params{};
  P.q = reinterpret_cast<const __half*>(q);
  P.bal = ck ? nullptr : c->balancer;  // per-channel keys are not balanced (FP16 important tier)
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
  int n_pend = 0;
  if (ck) {  // closed groups in the low tier's splits, the waiting pairs in one more CTA
    n_pend = c->n_lo % kGS;
    P.lo.n = c->n_lo - n_pend;
    P.pend = TierPtrs{static_cast<const uint8_t*>(c->k_pend), static_cast<const uint8_t*>(c->v_pend), nullptr,
                      nullptr, kGS, n_pend};
  }
  P.nsplit_lo = (P.lo.n + pl.chunk_lo - 1) / pl.chunk_lo;
  const DecWs wl = dec_ws_layout(c);
  P.smax = wl.smax;
  P.hi_logits = hi_logits;
  char* wsb = static_cast<char*>(ws);
  P.ws_o = reinterpret_cast<float*>(wsb + wl.o);
  P.ws_ml = reinterpret_cast<float*>(wsb + wl.ml);
  P.qf_out = reinterpret_cast<uint32_t*>(wsb + wl.qf);
  P.qf = P.qf_out;
  P.qc = ck ? reinterpret_cast<float*>(wsb + wl.qc) : nullptr;
  nsplit = P.nsplit_hi + P.nsplit_lo + (n_pend > 0 ? 1 : 0);
  if (nsplit < 1) return fail(MIKV_ESHAPE, "%s: nothing to attend", who);
  const int fmt = c->hi_bits * 100 + c->lo_bits;
  if (fmt != 1602 && fmt != 1604 && fmt != 1608 && fmt != 802 && fmt != 804 && fmt != 808 &&
      fmt != 402 && fmt != 404)
    return fail(MIKV_EUNSUPPORTED, "%s: bits %d/%d", who, c->hi_bits, c->lo_bits);
  return MIKV_OK;
}

// after: the kernel launched just before on `s` is one of ours; step: the decode step's
// token append, launched together with the query prep
int launch_partials(const Params& P, const mikv_cache* c, int nsplit, cudaStream_t s, bool after,
                    const AppendArgs* step) {
  const dim3 grid(nsplit, c->B * c->Hkv);
  if (c->key_mode == MIKV_KEYS_PER_CHANNEL)
    return c->lo_bits == 2 ? launch_nt<16, 2, true>(P, grid, s, after, step)
                           : launch_nt<16, 4, true>(P, grid, s, after, step);
  int e;
  switch (c->hi_bits * 100 + c->lo_bits) {
    case 1602: e = launch_nt<16, 2>(P, grid, s, after, step); break;
    case 1604: e = launch_nt<16, 4>(P, grid, s, after, step); break;
    case 1608: e = launch_nt<16, 8>(P, grid, s, after, step); break;
    case 802: e = launch_nt<8, 2>(P, grid, s, after, step); break;
    case 804: e = launch_nt<8, 4>(P, grid, s, after, step); break;
    case 402: e = launch_nt<4, 2>(P, grid, s, after, step); break;
    case 404: e = launch_nt<4, 4>(P, grid, s, after, step); break;
    default: e = launch_nt<8, 8>(P, grid, s, after, step); break;
  }
  return e;
}

int n_keep_of(int L, int pct, int window) {
  const long p = static_cast<long>(pct) * L / 100;
  return static_cast<int>(std::min<long>(L, std::max<long>(window, p)));
}
}  // namespace
}  // namespace mikv

extern "C" int mikv_set_attention_events(void* begin, void* end) {
  clear_error();
  if ((begin == nullptr) != (end == nullptr))
    return fail(MIKV_EINVAL, "set_attention_events: give both events or neither");
  t_ev_begin = static_cast<cudaEvent_t>(begin);
  t_ev_end = static_cast<cudaEvent_t>(end);
  return MIKV_OK;
}

extern "C" int mikv_decode_attention(const uint16_t* q, const mikv_cache* c, float* out,
                                     float* lse, float* hi_logits, void* ws, size_t ws_bytes,
                                     void* stream) {
  clear_error();
  if (int e = validate_cache_public(c, "decode_attention")) return e;
  if (!q || !out || !lse || !ws) return fail(MIKV_EINVAL, "decode_attention: null pointer");
  Params P;
  int nsplit = 0;
  if (int e = prepare_decode(q, c, hi_logits, ws, ws_bytes, P, nsplit, "decode_attention")) return e;
  cudaStream_t s = as_stream(stream);
  if (int e = launch_partials(P, c, nsplit, s, false, nullptr)) return e;
  return check_launch_after(
      launch_after(decode_merge_kernel, dim3(c->B * c->Hq * merge_chunks(nsplit)),
                   dim3(kD * merge_groups(nsplit) / merge_chunks(nsplit)), 0, s,
                   P.ws_o, P.ws_ml, P.smax, nsplit, out, lse),
      "decode_merge_kernel");
}

namespace mikv {
namespace {
// Step workspace after the attention workspace: per-head logits of the important tier, then
// per-chunk victim candidates (score, position, slot) and one ticket per (batch, key head).
struct StepWs {
  size_t logits, cand_s, cand_p, cand_j, ticket, total;
};
StepWs step_ws_layout(const mikv_cache* c, size_t dec_ws) {
  const size_t units = static_cast<size_t>(c->B) * c->Hkv;
  const size_t nchunk = std::max<size_t>(1, (static_cast<size_t>(c->cap_hi) + kEpiChunk - 1) / kEpiChunk);
  StepWs w;
  w.logits = dec_ws;
  w.cand_s = w.logits + align_up(static_cast<size_t>(c->B) * c->Hq * c->cap_hi * sizeof(float), 256);
  w.cand_p = w.cand_s + align_up(units * nchunk * sizeof(float), 256);
  w.cand_j = w.cand_p + align_up(units * nchunk * sizeof(int), 256);
  w.ticket = w.cand_j + align_up(units * nchunk * sizeof(int), 256);
  w.total = w.ticket + align_up(units * sizeof(unsigned), 256);
  return w;
}
}  // namespace
}  // namespace mikv

extern "C" size_t mikv_decode_step_workspace_bytes(const mikv_cache* c) {
  const size_t a = mikv_decode_workspace_bytes(c);
  if (a == 0) return 0;
  return step_ws_layout(c, a).total;
}

extern "C" int mikv_decode_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                int pos, int budget_pct, int window, int policy, mikv_cache* c,
                                float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (int e = validate_cache_public(c, "decode_step")) return e;
  if (!q || !k_new || !v_new || !out || !lse || !ws) return fail(MIKV_EINVAL, "decode_step: null pointer");
  if (policy != MIKV_H2O && policy != MIKV_CRITICALKV) return fail(MIKV_EINVAL, "decode_step: policy %d", policy);
  if (pos < 0 || budget_pct < 0 || budget_pct > 100 || window < 0)
    return fail(MIKV_ESHAPE, "decode_step: pos=%d budget_pct=%d window=%d", pos, budget_pct, window);
  if (c->n_hi + 1 > c->cap_hi) return fail(MIKV_ESHAPE, "decode_step: important tier full (%d)", c->cap_hi);
  if ((c->cap_hi + kEpiChunk - 1) / kEpiChunk > 65535)
    return fail(MIKV_EUNSUPPORTED, "decode_step: cap_hi %d above %d", c->cap_hi, 65535 * kEpiChunk);
  const size_t need = mikv_decode_step_workspace_bytes(c);
  if (ws_bytes < need) return fail(MIKV_ESHAPE, "decode_step: workspace %zu < %zu", ws_bytes, need);
  const int L = pos + 1;
  const bool demote = policy == MIKV_H2O && c->n_hi + 1 > n_keep_of(L, budget_pct, window);
  mikv_cache after = *c;  // counts once the new token is appended
  after.n_hi += 1;
  DemoteArgs da;
  if (int e = demote_args(&after, nullptr, da)) {
    if (demote) return e;
    da = DemoteArgs{};
    da.cap_hi = after.cap_hi;
    da.n_hi = after.n_hi;
    da.scores = after.scores;
    da.pos_hi = after.pos_hi;
  }
  const size_t dec_ws = mikv_decode_workspace_bytes(c);
  const StepWs wl = step_ws_layout(c, dec_ws);
  char* wsb = static_cast<char*>(ws);
  float* logits = reinterpret_cast<float*>(wsb + wl.logits);
  Params P;
  int nsplit = 0;
  if (int e = prepare_decode(q, &after, logits, ws, dec_ws, P, nsplit, "decode_step")) return e;
  cudaStream_t s = as_stream(stream);
  unsigned* ticket = reinterpret_cast<unsigned*>(wsb + wl.ticket);
  // 1.+2. one launch appends the new token to the important tier at slot n_hi (position pos,
  //    score 0), clears the demotion tickets and prepares the query fragments; then the
  //    split-K attention over both tiers
  AppendArgs aa;
  if (int e = append_args(true, k_new, v_new, 1, nullptr, 1, pos, nullptr, c, ticket, aa)) return e;
  if (int e = launch_partials(P, &after, nsplit, s, true, &aa)) return e;
  c->n_hi += 1;
  // 3. merge
  if (int e = check_launch_after(
          launch_after(decode_merge_kernel, dim3(c->B * c->Hq * merge_chunks(nsplit)),
                       dim3(kD * merge_groups(nsplit) / merge_chunks(nsplit)), 0,
                       s, P.ws_o, P.ws_ml, P.smax, nsplit, out, lse),
          "decode_merge_kernel"))
    return e;
  // 4. score update + demotion
  const int rep = c->Hq / c->Hkv;
  EpiArgs ea{};
  ea.logits = logits;
  ea.lse = lse;
  ea.Hq = c->Hq;
  ea.Hkv = c->Hkv;
  ea.nchunk = std::max(1, (after.n_hi + kEpiChunk - 1) / kEpiChunk);
  ea.demote = demote ? 1 : 0;
  ea.limit = L - window;
  ea.da = da;
  ea.cand_s = reinterpret_cast<float*>(wsb + wl.cand_s);
  ea.cand_p = reinterpret_cast<int*>(wsb + wl.cand_p);
  ea.cand_j = reinterpret_cast<int*>(wsb + wl.cand_j);
  ea.ticket = ticket;
  const dim3 egrid(c->B * c->Hkv, ea.nchunk);
  cudaError_t err;
  switch (rep) {
    case 1: err = launch_after(decode_score_demote_kernel<1>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 2: err = launch_after(decode_score_demote_kernel<2>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 3: err = launch_after(decode_score_demote_kernel<3>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 4: err = launch_after(decode_score_demote_kernel<4>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 5: err = launch_after(decode_score_demote_kernel<5>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 6: err = launch_after(decode_score_demote_kernel<6>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    case 7: err = launch_after(decode_score_demote_kernel<7>, egrid, dim3(kEpiThreads), 0, s, ea); break;
    default: err = launch_after(decode_score_demote_kernel<8>, egrid, dim3(kEpiThreads), 0, s, ea); break;
  }
  if (int e = check_launch_after(err, "decode_score_demote_kernel")) return e;
  if (demote) {
    c->n_hi -= 1;
    c->n_lo += 1;
    // per-channel keys: the demoted pair was the 64th waiting one, so its group closes
    if (c->key_mode == MIKV_KEYS_PER_CHANNEL && c->n_lo % kGS == 0) return channel_close_waiting(c, s);
  }
  return MIKV_OK;
}
