// K2: per-token asymmetric group quantisation and append into a cache tier, and
// the demotion of one important-tier slot into the low-bit tier.
//
// Sources: "No Token Left Behind" reading notes (velog), "Key contributions 1)"
// (evicted KV kept with per-token asymmetric quantisation, LLM-QAT), "2)" (keys
// quantised as I(k*b); group size = half the head dimension), "3)" (INT8
// important tier).
//
// Appends of many tokens (prefill) run append_tile_kernel below: 32 tokens of one (batch, key
// head) per CTA, one thread per (tensor, 64-channel group, token).  The one-token paths
// (demotion, and the decode step's own append) keep one warp per (token, key head): lane l
// owns channels 4l..4l+3, so a group is one half-warp and its min/max are two 4-step shuffle
// reductions.  Every step takes round-to-nearest in the order the format fixes:
//   x = fl(k*b) (keys of a quantised tier) or v
//   s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn)
//   code = clamp(rint_even(fl(fl(x - z) / s)), 0, qmax); 0 where s == 0.
// Codes are packed LSB-first (channel c at bit c*bits of the row), meta is the
// fp16 pair (scale, zero) per group.  HBM-bound: 512 B read per token-head,
// 80/144/272/512 B written.
#include <algorithm>

#include "quant_device.cuh"

namespace mikv {
namespace {

// Appends of many tokens (prefill): one CTA of 128 threads per (32 consecutive tokens of the
// append, unit).  The 32 source rows of K and V are gathered with coalesced 16-byte loads into
// shared memory (16-byte chunk c of row r at chunk c ^ (r % 8), so that the eight rows a
// quarter-warp reads next sit in different banks); then thread (tensor, group, row) quantises
// one 64-channel group of one row from there and stores its codes with 16-byte stores:
// 16 / 32 / 64 bytes for INT2 / INT4 / INT8.  An FP16 tier is a plain 16-byte copy.
constexpr int kTileTok = 32;
constexpr int kTileThreads = 128;

// Packed fp32 pairs (explicit round-to-nearest PTX) for the steps after the balancer product.
__device__ __forceinline__ uint64_t f2_bits(float2 a) {
  return static_cast<uint64_t>(__float_as_uint(a.x)) | (static_cast<uint64_t>(__float_as_uint(a.y)) << 32);
}
__device__ __forceinline__ float2 bits_f2(uint64_t u) {
  return make_float2(__uint_as_float(static_cast<uint32_t>(u)), __uint_as_float(static_cast<uint32_t>(u >> 32)));
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

// Chunk `chunk` (8 channels) of a shared-memory row as 4 fp32 pairs, times the per-channel
// factors `mul` (the balancer for keys, ones for values: x * 1 is exact).  The product is
// taken with scalar __fmul_rn, which is never merged into a fused multiply-add: fl(k * b) - z
// must be rounded twice, as the format states.  A packed multiply whose only use was the
// packed subtraction of z came out fused on sm_103a (one rounding of k * b - z), which moved
// exact ties such as d / s = 139.5 to 139.49998 and changed their codes.
__device__ __forceinline__ void chunk_f32x2(const uint8_t* row, int chunk, int r, const float* mul, float2 (&x)[4]) {
  const uint4 w = *reinterpret_cast<const uint4*>(row + ((chunk ^ (r & 7)) * 16));
  const __half2* h = reinterpret_cast<const __half2*>(&w);
  const float4 b0 = reinterpret_cast<const float4*>(mul)[2 * chunk];
  const float4 b1 = reinterpret_cast<const float4*>(mul)[2 * chunk + 1];
  const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h[e]);
    x[e] = make_float2(__fmul_rn(f.x, bb[2 * e]), __fmul_rn(f.y, bb[2 * e + 1]));
  }
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// rint_even(fl(d / s)) with the correctly rounded division, for values near a tie.
__device__ __noinline__ float rint_div(float d, float s) { return rintf(__fdiv_rn(d, s)); }

// Codes and meta of one 64-channel group of one row (8 swizzled 16-byte chunks in shared
// memory).  code = clamp(rint_even(fl(d / s)), 0, qmax), d = fl(x - z), is computed from
// r = fl(1/s), taken once per group (__frcp_rn is correctly rounded), as q0 = fl(d * r).  q0 is
// within a relative 2^-23 (1 + 2^-24) of d / s: below |d/s| = 257 that is less than 2^-14
// absolute, and fl(d / s) is within 2^-16 of d / s, so rint(q0) and rint(fl(d / s)) can only
// differ when d / s lies within ~2^-13 of a half-integer.  A value whose q0 comes within
// 2^-12 of one (|q0 - rint(q0)| > 1/2 - 2^-12) takes the correctly rounded __fdiv_rn quotient
// instead.  The codes therefore equal the rounding of fl(d / s) in every case.
//   d and q0 are monotone in x, so when the group's extremes give q0 inside
// (-1/2, qmax + 1/2) with a 2^-10 margin, no value needs the clamp: that common case runs on
// packed fp32 pairs, rounds with 1.5 * 2^23 (q + 1.5*2^23 lands on the integer grid, ties to
// even, for |q| < 2^22) and packs the codes of 16-bit fields as exact fp32 sums
// sum c_i 2^(BITS i) < 2^16.  Otherwise every value is clamped one by one.
constexpr float kTieGuard = 1.f / 4096.f;
constexpr float kRangeGuard = 1.f / 1024.f;
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23

template <int BITS>
__device__ __forceinline__ uint32_t quantize_group64(const uint8_t* row, int g, int r, const float* mul,
                                                     bool scaled, uint32_t (&out)[64 * BITS / 32]) {
  constexpr int kWords = 64 * BITS / 32;
  constexpr int qmax = (1 << BITS) - 1;
  float mn, mx;
  if (scaled) {  // keys of a balanced tier: the extremes of fl(k * b)
    mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 x[4];
      chunk_f32x2(row, g * 8 + i, r, mul, x);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        mn = min3f(mn, x[p].x, x[p].y);
        mx = max3f(mx, x[p].x, x[p].y);
      }
    }
  } else {  // fp16 values as they are: min / max of fp16 numbers are exact in half2 arithmetic
    __half2 m0 = __float2half2_rn(INFINITY), m1 = __float2half2_rn(-INFINITY);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 w = *reinterpret_cast<const uint4*>(row + (((g * 8 + i) ^ (r & 7)) * 16));
      const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        m0 = __hmin2(m0, h[e]);
        m1 = __hmax2(m1, h[e]);
      }
    }
    mn = fminf(__low2float(m0), __high2float(m0));
    mx = fmaxf(__low2float(m1), __high2float(m1));
  }
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(qmax));
  const __half sh = __float2half_rn(s32), zh = __float2half_rn(mn);
  const float sf = __half2float(sh), zf = __half2float(zh);
#pragma unroll
  for (int k = 0; k < kWords; ++k) out[k] = 0u;
  if (sf == 0.f) return pack_half2(sh, zh);
  const float rf = __frcp_rn(sf);
  const float q_lo = __fmul_rn(__fsub_rn(mn, zf), rf), q_hi = __fmul_rn(__fsub_rn(mx, zf), rf);
  if (q_lo > -0.5f + kRangeGuard && q_hi < qmax + 0.5f - kRangeGuard) {
    const float2 nz = make_float2(-zf, -zf), r2 = make_float2(rf, rf);
    const float2 mg = make_float2(kRoundMagic, kRoundMagic), nmg = make_float2(-kRoundMagic, -kRoundMagic);
    const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 x[4], d[4], qi[4];
      chunk_f32x2(row, g * 8 + i, r, mul, x);
      float emax = 0.f;  // largest |q0 - rint(q0)| of the chunk
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        d[p] = add2_rn(x[p], nz);
        const float2 q = mul2_rn(d[p], r2);
        qi[p] = add2_rn(add2_rn(q, mg), nmg);
        const float2 e = __ffma2_rn(qi[p], m1, q);  // q - qi, exact
        emax = max3f(emax, fabsf(e.x), fabsf(e.y));
      }
      if (emax > 0.5f - kTieGuard) {  // rare: a value of this chunk is near a tie
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if (fabsf(__fmul_rn(d[p].x, rf) - qi[p].x) > 0.5f - kTieGuard) qi[p].x = rint_div(d[p].x, sf);
          if (fabsf(__fmul_rn(d[p].y, rf) - qi[p].y) > 0.5f - kTieGuard) qi[p].y = rint_div(d[p].y, sf);
        }
      }
      // 16-bit fields of kPack codes each, summed exactly as fp32 pairs
      constexpr int kPack = 16 / BITS;
#pragma unroll
      for (int f = 0; f < 8 / kPack; ++f) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = f * kPack / 2; p < (f + 1) * kPack / 2; ++p) {
          const int e0 = 2 * p - f * kPack;  // index of qi[p].x within the field
          acc = __ffma2_rn(qi[p], make_float2(static_cast<float>(1 << (BITS * e0)),
                                              static_cast<float>(1 << (BITS * (e0 + 1)))), acc);
        }
        const int bit = (i * 8 + f * kPack) * BITS;  // first bit of the field in the group
        out[bit / 32] |= (__float_as_uint((acc.x + acc.y) + 8388608.f) & 0xffffu) << (bit % 32);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 x[4];
      chunk_f32x2(row, g * 8 + i, r, mul, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xe = e & 1 ? x[e >> 1].y : x[e >> 1].x;
        const float d = __fsub_rn(xe, zf);
        const float q = __fmul_rn(d, rf);
        float qi = rintf(q);
        if (fabsf(q - qi) > 0.5f - kTieGuard) qi = rint_div(d, sf);
        const int ch = i * 8 + e;
        out[ch * BITS / 32] |= static_cast<uint32_t>(fminf(fmaxf(qi, 0.f), static_cast<float>(qmax)))
                               << ((ch * BITS) % 32);
      }
    }
  }
  return pack_half2(sh, zh);
}

// Tile of 32 consecutive tokens of one unit: 2 tensors x 32 rows x 16 chunks of 16 bytes,
// kPer chunks per thread (rows (t / 16) + 8 m, chunk t % 16).
constexpr int kPer = 2 * kTileTok * 16 / kTileThreads;

struct TileAt {
  long unit;
  int j0, nt;
};
__device__ __forceinline__ TileAt tile_at(const AppendArgs& a, long tile, int tiles_per_unit) {
  TileAt p;
  p.unit = tile / tiles_per_unit;
  p.j0 = static_cast<int>(tile % tiles_per_unit) * kTileTok;
  p.nt = min(kTileTok, a.n_tokens - p.j0);
  return p;
}
// Source row of token j0 + r of the tile, or -1 (past the end, or out of range: left unchanged).
__device__ __forceinline__ int tile_src(const AppendArgs& a, const TileAt& p, int r) {
  if (r >= p.nt) return -1;
  const int src = a.src_pos ? a.src_pos[p.unit * a.n_tokens + p.j0 + r] : p.j0 + r;
  return (src < 0 || src >= a.src_len) ? -1 : src;
}

// FP16 tier: a plain copy, all of a thread's 16-byte loads issued before its stores.
__global__ void __launch_bounds__(kTileThreads) append_copy_kernel(AppendArgs a, int tiles_per_unit) {
  const TileAt p = tile_at(a, blockIdx.x, tiles_per_unit);
  const int t = threadIdx.x, c = t & 15;
  int src[kPer / 2];
  uint4 w[kPer];
#pragma unroll
  for (int m = 0; m < kPer / 2; ++m) src[m] = tile_src(a, p, (t >> 4) + 8 * m);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int m = k % (kPer / 2), tensor = k / (kPer / 2);
    if (src[m] >= 0) w[k] = __ldg(reinterpret_cast<const uint4*>((tensor ? a.v : a.k) + (p.unit * a.src_len + src[m]) * kD) + c);
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int m = k % (kPer / 2), tensor = k / (kPer / 2), r = (t >> 4) + 8 * m;
    if (src[m] >= 0)
      reinterpret_cast<uint4*>((tensor ? a.dv : a.dk) + (p.unit * a.cap + a.base_slot + p.j0 + r) * (kD * 2))[c] = w[k];
  }
  if (t < kTileTok) {
    const int sr = tile_src(a, p, t);
    if (sr >= 0) {
      const long slot = p.unit * a.cap + a.base_slot + p.j0 + t;
      a.dpos[slot] = sr + a.pos_base;
      if (a.dscores) a.dscores[slot] = a.src_scores ? a.src_scores[p.unit * a.n_tokens + p.j0 + t] : 0.f;
    }
  }
}

// Quantised tiers: one CTA per tile.  Its rows (and the unit's balancer) are copied into
// shared memory with cp.async, all of a thread's copies in flight at once; then thread
// (tensor, group, row) quantises one group.  Several CTAs per SM overlap one tile's copies
// with another's arithmetic.
template <int BITS>
__global__ void __launch_bounds__(kTileThreads) append_tile_kernel(AppendArgs a, int tiles_per_unit) {
  __shared__ __align__(16) uint8_t rows[2][kTileTok][kD * 2];
  __shared__ __align__(16) float smul[2][kD];  // keys: the balancer (or ones); values: ones
  __shared__ int ssrc[kTileTok];
  const int t = threadIdx.x, c = t & 15;
  const TileAt p = tile_at(a, blockIdx.x, tiles_per_unit);
#pragma unroll
  for (int m = 0; m < kPer / 2; ++m) {
    const int r = (t >> 4) + 8 * m;
    const int src = tile_src(a, p, r);
    if (c == 0) ssrc[r] = src;
#pragma unroll
    for (int tensor = 0; tensor < 2; ++tensor) {
      const __half* row = (tensor ? a.v : a.k) + (p.unit * a.src_len + (src >= 0 ? src : 0)) * kD;
      cp_async16(smem_u32(&rows[tensor][r][(c ^ (r & 7)) * 16]), row + c * 8, src >= 0);
    }
  }
  if (a.bal && t < kD / 4) cp_async16(smem_u32(&smul[0][4 * t]), a.bal + p.unit * kD + 4 * t, true);
  if (!a.bal) smul[0][t] = 1.f;
  smul[1][t] = 1.f;
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (t < kTileTok && ssrc[t] >= 0) {
    const long slot = p.unit * a.cap + a.base_slot + p.j0 + t;
    a.dpos[slot] = ssrc[t] + a.pos_base;
    if (a.dscores) a.dscores[slot] = a.src_scores ? a.src_scores[p.unit * a.n_tokens + p.j0 + t] : 0.f;
  }
  const int tensor = t >> 6, g = (t >> 5) & 1, r = t & 31;
  if (ssrc[r] < 0) return;
  uint32_t out[64 * BITS / 32];
  const uint32_t meta = quantize_group64<BITS>(rows[tensor][r], g, r, smul[tensor], tensor == 0 && a.bal != nullptr, out);
  const long slot = p.unit * a.cap + a.base_slot + p.j0 + r;
  constexpr int kRB = kD * BITS / 8;
  uint8_t* dst = (tensor ? a.dv : a.dk) + slot * kRB + g * (kRB / 2);
#pragma unroll
  for (int k = 0; k < 64 * BITS / 128; ++k)
    reinterpret_cast<uint4*>(dst)[k] = make_uint4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
  reinterpret_cast<uint32_t*>(tensor ? a.dvm : a.dkm)[slot * 2 + g] = meta;
}

// ---------------------------------------------------------------------------------
// Per-channel keys ([notes] Appendix C remarks; [paperlayer] C: group 64, keys per channel):
// closing groups of 64 retained pairs.  Keys: per channel c, the per-token quantizer's rule
// over the group's 64 values of c (s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn),
// code = clamp(rint_even(fl(fl(x - z) / s)), 0, qmax)), codes into the per-token rows (channel
// c at bit c * bits), (s, z) into the group's meta row [D]; values: per token, as the
// per-token tier.  No balancer.
struct ChanArgs {
  const __half* k;         // prefill: source [units][src_len][D]; closing: the waiting buffer
  const __half* v;
  const int32_t* src_pos;  // prefill: [units][n_tokens]; closing: null (rows 0 .. 63 in order)
  long src_stride;         // rows per unit in k / v (src_len, or 64 for the buffer)
  int src_len, n_tokens, pos_base;
  int base_slot;           // first low-tier slot written (a multiple of 64)
  int cap_lo, ngroups;     // full groups to close; a prefill's tail goes to the waiting buffer
  uint8_t* k_lo;
  uint8_t* v_lo;
  __half2* k_meta;         // [units][cap_lo / 64][D]
  __half2* v_meta;         // [units][cap_lo][2]
  int32_t* pos_lo;         // written by a prefill (closing: positions are already in place)
  __half* k_pend;          // [units][64][D]
  __half* v_pend;
};

// CTA (group gi, unit), 128 threads.  gi < ngroups: gather the group's 64 key and value rows
// (cp.async, 16 bytes), thread c quantises key channel c over the 64 rows (column extremes,
// codes into a shared byte matrix), thread (row, half) quantises one value group of a row;
// rows of key codes are packed at the end.  gi == ngroups (prefill only): the tail rows are
// copied to the waiting buffer.  VALUES false: keys only (the standalone group quantiser).
template <int BITS, bool VALUES = true>
__global__ void __launch_bounds__(kTileThreads) channel_close_kernel(ChanArgs a) {
  __shared__ __align__(16) __half ks[kGS][kD];        // keys, row-major
  __shared__ __align__(16) uint8_t vs[VALUES ? kGS : 1][kD * 2];  // values, 16-byte chunks swizzled by row
  __shared__ __align__(16) uint8_t cs[kGS][kD];       // key codes
  __shared__ __half2 ext[2][kD / 2][2];                // per row half: (min, max) of channel pairs
  __shared__ __align__(16) float ones[kD];
  __shared__ int ssrc[kGS];
  const long unit = blockIdx.y;
  const int gi = blockIdx.x, t = threadIdx.x;
  const int j0 = gi * kGS;                               // first token of this CTA
  const int nrow = min(kGS, a.n_tokens - j0);
  if (t < kGS) {
    int src = -1;
    if (t < nrow) {
      src = a.src_pos ? a.src_pos[unit * a.n_tokens + j0 + t] : j0 + t;
      if (src < 0 || src >= a.src_len) src = -1;
    }
    ssrc[t] = src;
    if (a.src_pos && src >= 0) a.pos_lo[unit * a.cap_lo + a.base_slot + j0 + t] = src + a.pos_base;
  }
  ones[t] = 1.f;
  __syncthreads();
  if (gi >= a.ngroups) {  // prefill tail: rows wait unquantised in buffer rows 0 .. nrow - 1
    for (int i = t; i < nrow * 16 * 2; i += kTileThreads) {
      const int tensor = i / (nrow * 16), r = (i >> 4) % nrow, c = i & 15;
      const int src = ssrc[r];
      if (src < 0) continue;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>((tensor ? a.v : a.k) + (unit * a.src_stride + src) * kD) + c);
      reinterpret_cast<uint4*>((tensor ? a.v_pend : a.k_pend) + (unit * kGS + r) * kD)[c] = w;
    }
    return;
  }
  // gather: 2 tensors x 64 rows x 16 chunks, 16 per thread, all in flight together
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int r = (t >> 4) + 8 * m, c = t & 15;
    const int src = ssrc[r];
    const long off = (unit * a.src_stride + (src >= 0 ? src : 0)) * kD + c * 8;
    cp_async16(smem_u32(&ks[r][c * 8]), a.k + off, src >= 0);
    if (VALUES) cp_async16(smem_u32(&vs[r][(c ^ (r & 7)) * 16]), a.v + off, src >= 0);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  constexpr int qmax = (1 << BITS) - 1;
  {  // key channels (2 cp, 2 cp + 1), cp = t % 64, over rows 32 h .. 32 h + 31, h = t / 64: the
     // pair's extremes in half2 arithmetic (exact), combined with the other half through shared
     // memory, then the codes on packed fp32 pairs (the same quotient rule as the per-token tiers)
    const int cp = t & 63, h = t >> 6, c = 2 * cp;
    __half2 lo2 = __float2half2_rn(INFINITY), hi2 = __float2half2_rn(-INFINITY);
#pragma unroll 8
    for (int r = 32 * h; r < 32 * h + 32; ++r) {
      const __half2 x = *reinterpret_cast<const __half2*>(&ks[r][c]);
      lo2 = __hmin2(lo2, x);
      hi2 = __hmax2(hi2, x);
    }
    ext[h][cp][0] = lo2;
    ext[h][cp][1] = hi2;
    __syncthreads();
    lo2 = __hmin2(ext[0][cp][0], ext[1][cp][0]);
    hi2 = __hmax2(ext[0][cp][1], ext[1][cp][1]);
    const float2 mn = __half22float2(lo2), mx = __half22float2(hi2);
    const float s0 = __fdiv_rn(__fsub_rn(mx.x, mn.x), static_cast<float>(qmax));
    const float s1 = __fdiv_rn(__fsub_rn(mx.y, mn.y), static_cast<float>(qmax));
    const __half sh0 = __float2half_rn(s0), zh0 = __float2half_rn(mn.x);
    const __half sh1 = __float2half_rn(s1), zh1 = __float2half_rn(mn.y);
    const float sf0 = __half2float(sh0), zf0 = __half2float(zh0), sf1 = __half2float(sh1), zf1 = __half2float(zh1);
    const float rf0 = sf0 != 0.f ? __frcp_rn(sf0) : 0.f, rf1 = sf1 != 0.f ? __frcp_rn(sf1) : 0.f;
    if (h == 0) {
      __half2* km = a.k_meta + (unit * (a.cap_lo / kGS) + (a.base_slot + j0) / kGS) * kD + c;
      km[0] = __halves2half2(sh0, zh0);
      km[1] = __halves2half2(sh1, zh1);
    }
    // extremes' quotients: inside (-1/2, qmax + 1/2) no value of the channel needs the clamp
    const bool fast = sf0 != 0.f && sf1 != 0.f &&
                      __fmul_rn(__fsub_rn(mn.x, zf0), rf0) > -0.5f + kRangeGuard &&
                      __fmul_rn(__fsub_rn(mx.x, zf0), rf0) < qmax + 0.5f - kRangeGuard &&
                      __fmul_rn(__fsub_rn(mn.y, zf1), rf1) > -0.5f + kRangeGuard &&
                      __fmul_rn(__fsub_rn(mx.y, zf1), rf1) < qmax + 0.5f - kRangeGuard;
    if (fast) {
      const float2 nz = make_float2(-zf0, -zf1), r2 = make_float2(rf0, rf1);
      const float2 mg = make_float2(kRoundMagic, kRoundMagic), nmg = make_float2(-kRoundMagic, -kRoundMagic);
#pragma unroll 4
      for (int r = 32 * h; r < 32 * h + 32; ++r) {
        const float2 d = add2_rn(__half22float2(*reinterpret_cast<const __half2*>(&ks[r][c])), nz);
        const float2 q = mul2_rn(d, r2);
        float2 qi = add2_rn(add2_rn(q, mg), nmg);
        const float2 e = __ffma2_rn(qi, make_float2(-1.f, -1.f), q);  // q - qi, exact
        if (fmaxf(fabsf(e.x), fabsf(e.y)) > 0.5f - kTieGuard) {       // rare: near a tie
          if (fabsf(e.x) > 0.5f - kTieGuard) qi.x = rint_div(d.x, sf0);
          if (fabsf(e.y) > 0.5f - kTieGuard) qi.y = rint_div(d.y, sf1);
        }
        *reinterpret_cast<uint16_t*>(&cs[r][c]) =
            static_cast<uint16_t>((__float_as_uint(qi.x + 8388608.f) & 0xffu) |
                                  ((__float_as_uint(qi.y + 8388608.f) & 0xffu) << 8));
      }
    } else {  // a constant channel (scale 0: codes 0), or one whose extremes need the clamp
#pragma unroll 4
      for (int r = 32 * h; r < 32 * h + 32; ++r) {
        const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&ks[r][c]));
        uint32_t code[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float sf = e ? sf1 : sf0, zf = e ? zf1 : zf0, rf = e ? rf1 : rf0;
          if (sf != 0.f) {
            const float d = __fsub_rn(e ? x.y : x.x, zf);
            const float q = __fmul_rn(d, rf);
            float qi = rintf(q);
            if (fabsf(q - qi) > 0.5f - kTieGuard) qi = rint_div(d, sf);  // near a tie: exact quotient
            code[e] = static_cast<uint32_t>(fminf(fmaxf(qi, 0.f), static_cast<float>(qmax)));
          }
        }
        *reinterpret_cast<uint16_t*>(&cs[r][c]) = static_cast<uint16_t>(code[0] | (code[1] << 8));
      }
    }
  }
  if (VALUES) {  // value group (t >> 6) of row t % 64, per token
    const int r = t & 63, g = t >> 6;
    uint32_t out[64 * BITS / 32];
    const uint32_t meta = quantize_group64<BITS>(vs[r], g, r, ones, false, out);
    const long slot = unit * a.cap_lo + a.base_slot + j0 + r;
    constexpr int kRB = kD * BITS / 8;
    uint8_t* dst = a.v_lo + slot * kRB + g * (kRB / 2);
#pragma unroll
    for (int k = 0; k < 64 * BITS / 128; ++k)
      reinterpret_cast<uint4*>(dst)[k] = make_uint4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
    reinterpret_cast<uint32_t*>(a.v_meta)[slot * 2 + g] = meta;
  }
  __syncthreads();
  {  // pack the key code rows: thread (row t % 64, half t / 64) packs 64 channels
    const int r = t & 63, half = t >> 6;
    constexpr int kPer = 32 / BITS;             // codes per 32-bit word
    constexpr int kW = 64 / kPer;               // words per half row
    uint32_t w[kW];
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) x |= static_cast<uint32_t>(cs[r][half * 64 + i * kPer + e]) << (BITS * e);
      w[i] = x;
    }
    constexpr int kRB = kD * BITS / 8;
    uint8_t* dst = a.k_lo + (unit * a.cap_lo + a.base_slot + j0 + r) * kRB + half * (kRB / 2);
#pragma unroll
    for (int k = 0; k < kW / 4; ++k) reinterpret_cast<uint4*>(dst)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}

__global__ void __launch_bounds__(256) demote_kernel(DemoteArgs a) {
  const int lane = threadIdx.x & 31;
  const long unit = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (unit >= a.units) return;
  demote_one(a, unit, a.victim[unit], lane);
}

int validate_cache(const mikv_cache* c, const char* who) {
  if (!c) return fail(MIKV_EINVAL, "%s: null cache", who);
  if (c->D != kD) return fail(MIKV_EUNSUPPORTED, "%s: D=%d (only %d)", who, c->D, kD);
  if (c->hi_bits != 16 && c->hi_bits != 8 && c->hi_bits != 4)
    return fail(MIKV_EUNSUPPORTED, "%s: hi_bits=%d (16, 8 or 4)", who, c->hi_bits);
  if ((c->lo_bits != 2 && c->lo_bits != 4 && c->lo_bits != 8) || c->lo_bits > c->hi_bits)
    return fail(MIKV_EUNSUPPORTED, "%s: lo_bits=%d (2, 4 or 8, at most hi_bits)", who, c->lo_bits);
  if (c->B < 1 || c->Hkv < 1 || c->Hq < c->Hkv || c->Hq % c->Hkv || c->Hq / c->Hkv > 8)
    return fail(MIKV_ESHAPE, "%s: bad heads B=%d Hq=%d Hkv=%d", who, c->B, c->Hq, c->Hkv);
  if (c->cap_hi < 0 || c->cap_lo < 0 || c->n_hi < 0 || c->n_lo < 0 || c->n_hi > c->cap_hi ||
      c->n_lo > c->cap_lo)
    return fail(MIKV_ESHAPE, "%s: counts n_hi=%d/%d n_lo=%d/%d", who, c->n_hi, c->cap_hi, c->n_lo,
                c->cap_lo);
  if (c->key_mode != MIKV_KEYS_PER_TOKEN && c->key_mode != MIKV_KEYS_PER_CHANNEL)
    return fail(MIKV_EINVAL, "%s: key_mode %d", who, c->key_mode);
  if (c->key_mode == MIKV_KEYS_PER_CHANNEL) {
    if (c->hi_bits != 16 || (c->lo_bits != 2 && c->lo_bits != 4))
      return fail(MIKV_EUNSUPPORTED, "%s: per-channel keys need hi_bits 16 and lo_bits 2 or 4 (%d/%d)", who,
                  c->hi_bits, c->lo_bits);
    if (c->cap_lo % kGS) return fail(MIKV_ESHAPE, "%s: per-channel keys need cap_lo %% 64 == 0 (%d)", who, c->cap_lo);
    if (!c->k_pend || !c->v_pend) return fail(MIKV_EINVAL, "%s: null waiting-pair buffer", who);
    if (!aligned16(c->k_pend) || !aligned16(c->v_pend))
      return fail(MIKV_EALIGN, "%s: waiting-pair buffers must be 16-byte aligned", who);
  }
  return MIKV_OK;
}

}  // namespace

int validate_cache_public(const mikv_cache* c, const char* who) { return validate_cache(c, who); }

}  // namespace mikv

using namespace mikv;

namespace mikv {

// Validate an append of n_tokens source tokens into the HI or LO tier and fill its kernel
// arguments (counts in *c are not changed).  src_pos == nullptr means source token j goes
// to slot j.  ticket (optional): per-unit counters the kernel clears.
int append_args(bool hi, const uint16_t* k, const uint16_t* v, int src_len, const int32_t* src_pos,
                int n_tokens, int pos_base, const float* src_scores, const mikv_cache* c,
                unsigned* ticket, AppendArgs& a) {
  const long units = static_cast<long>(c->B) * c->Hkv;
  const int bits = hi ? c->hi_bits : c->lo_bits;
  if ((!k || !v) && n_tokens > 0) return fail(MIKV_EINVAL, "quantize_append: null k/v");
  if (n_tokens < 0 || src_len < 1) return fail(MIKV_ESHAPE, "quantize_append: n_tokens/src_len");
  const int base = hi ? c->n_hi : c->n_lo;
  const int cap = hi ? c->cap_hi : c->cap_lo;
  if (base + n_tokens > cap)
    return fail(MIKV_ESHAPE, "quantize_append: tier capacity %d exceeded (%d + %d)", cap, base,
                n_tokens);
  a = AppendArgs{};
  a.k = reinterpret_cast<const __half*>(k);
  a.v = reinterpret_cast<const __half*>(v);
  a.src_pos = src_pos;
  a.src_scores = src_scores;
  a.bal = (bits != 16) ? c->balancer : nullptr;
  a.Hkv = c->Hkv;
  a.src_len = src_len;
  a.n_tokens = n_tokens;
  a.pos_base = pos_base;
  a.cap = cap;
  a.base_slot = base;
  a.bits = bits;
  a.dk = static_cast<uint8_t*>(hi ? c->k_hi : c->k_lo);
  a.dv = static_cast<uint8_t*>(hi ? c->v_hi : c->v_lo);
  a.dkm = static_cast<__half2*>(hi ? c->k_hi_meta : c->k_lo_meta);
  a.dvm = static_cast<__half2*>(hi ? c->v_hi_meta : c->v_lo_meta);
  a.dpos = hi ? c->pos_hi : c->pos_lo;
  a.dscores = hi ? c->scores : nullptr;
  if (!a.dk || !a.dv || !a.dpos || (hi && !a.dscores))
    return fail(MIKV_EINVAL, "quantize_append: null tier buffer");
  if (bits != 16 && (!a.dkm || !a.dvm)) return fail(MIKV_EINVAL, "quantize_append: null meta");
  if (!aligned16(a.dk) || !aligned16(a.dv) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
      (bits != 16 && (!aligned16(a.dkm) || !aligned16(a.dvm))) || (a.bal && !aligned16(a.bal)))
    return fail(MIKV_EALIGN, "quantize_append: buffers must be 16-byte aligned");
  a.units_tokens = units * n_tokens;
  a.ticket = ticket;
  return MIKV_OK;
}

// Validate and launch an append (see append_args).
int append_tokens(bool hi, const uint16_t* k, const uint16_t* v, int src_len, const int32_t* src_pos,
                  int n_tokens, int pos_base, const float* src_scores, const mikv_cache* c,
                  cudaStream_t s) {
  AppendArgs a;
  if (int e = append_args(hi, k, v, src_len, src_pos, n_tokens, pos_base, src_scores, c, nullptr, a))
    return e;
  if (n_tokens == 0) return MIKV_OK;
  const long units = static_cast<long>(c->B) * c->Hkv;
  const int tiles_per_unit = (n_tokens + kTileTok - 1) / kTileTok;
  const long ntiles = units * tiles_per_unit;
  if (a.bits == 16) {
    if (ntiles > 0x7fffffffL) return fail(MIKV_ESHAPE, "quantize_append: %ld tiles", ntiles);
    append_copy_kernel<<<static_cast<unsigned>(ntiles), kTileThreads, 0, s>>>(a, tiles_per_unit);
    return check_launch("append_copy_kernel");
  }
  if (ntiles > 0x7fffffffL) return fail(MIKV_ESHAPE, "quantize_append: %ld tiles", ntiles);
  void (*kern)(AppendArgs, int) = a.bits == 8 ? append_tile_kernel<8>
                                  : a.bits == 4 ? append_tile_kernel<4> : append_tile_kernel<2>;
  kern<<<static_cast<unsigned>(ntiles), kTileThreads, 0, s>>>(a, tiles_per_unit);
  return check_launch("append_tile_kernel");
}

// Demotion arguments for the current counts of *c (victim list: [B*Hkv] hi slots).
int demote_args(const mikv_cache* c, const int32_t* victim, DemoteArgs& a) {
  if (c->n_hi < 1 || c->n_lo + 1 > c->cap_lo)
    return fail(MIKV_ESHAPE, "demotion: n_hi=%d n_lo=%d cap_lo=%d", c->n_hi, c->n_lo, c->cap_lo);
  a = DemoteArgs{};
  a.victim = victim;
  a.bal = c->balancer;
  a.units = c->B * c->Hkv;
  a.hi_bits = c->hi_bits;
  a.lo_bits = c->lo_bits;
  a.cap_hi = c->cap_hi;
  a.cap_lo = c->cap_lo;
  a.n_hi = c->n_hi;
  a.n_lo = c->n_lo;
  a.k_hi = static_cast<uint8_t*>(c->k_hi);
  a.v_hi = static_cast<uint8_t*>(c->v_hi);
  a.k_hi_meta = static_cast<__half2*>(c->k_hi_meta);
  a.v_hi_meta = static_cast<__half2*>(c->v_hi_meta);
  a.k_lo = static_cast<uint8_t*>(c->k_lo);
  a.v_lo = static_cast<uint8_t*>(c->v_lo);
  a.k_lo_meta = static_cast<__half2*>(c->k_lo_meta);
  a.v_lo_meta = static_cast<__half2*>(c->v_lo_meta);
  a.pos_hi = c->pos_hi;
  a.pos_lo = c->pos_lo;
  a.scores = c->scores;
  a.key_mode = c->key_mode;
  a.k_pend = static_cast<__half*>(c->k_pend);
  a.v_pend = static_cast<__half*>(c->v_pend);
  if (!a.k_hi || !a.v_hi || !a.k_lo || !a.v_lo || !a.k_lo_meta || !a.v_lo_meta || !a.pos_hi ||
      !a.pos_lo || !a.scores || (c->hi_bits != 16 && (!a.k_hi_meta || !a.v_hi_meta)))
    return fail(MIKV_EINVAL, "demotion: null cache buffer");
  if (!aligned16(a.k_hi) || !aligned16(a.v_hi) || !aligned16(a.k_lo) || !aligned16(a.v_lo) ||
      !aligned16(a.k_lo_meta) || !aligned16(a.v_lo_meta))
    return fail(MIKV_EALIGN, "demotion: buffers must be 16-byte aligned");
  return MIKV_OK;
}

ChanArgs chan_args(const mikv_cache* c) {
  ChanArgs a{};
  a.cap_lo = c->cap_lo;
  a.k_lo = static_cast<uint8_t*>(c->k_lo);
  a.v_lo = static_cast<uint8_t*>(c->v_lo);
  a.k_meta = static_cast<__half2*>(c->k_lo_meta);
  a.v_meta = static_cast<__half2*>(c->v_lo_meta);
  a.pos_lo = c->pos_lo;
  a.k_pend = static_cast<__half*>(c->k_pend);
  a.v_pend = static_cast<__half*>(c->v_pend);
  return a;
}

int launch_close(const ChanArgs& a, dim3 grid, int bits, cudaStream_t s) {
  if (bits == 2) channel_close_kernel<2><<<grid, kTileThreads, 0, s>>>(a);
  else channel_close_kernel<4><<<grid, kTileThreads, 0, s>>>(a);
  return check_launch("channel_close_kernel");
}

// The standalone per-channel group quantiser (mikv_channel_quantize): keys [units][n][D], the
// floor(n / 64) full groups of each unit quantised in place of rows, meta [units][n / 64][D].
int channel_quantize_keys(const __half* k, int units, int n, int bits, uint8_t* codes, __half2* meta,
                          cudaStream_t s) {
  const int ngrp = n / kGS;
  if (ngrp == 0) return MIKV_OK;  // every key is still waiting
  ChanArgs a{};
  a.k = k;
  a.src_stride = n;
  a.src_len = n;
  a.n_tokens = ngrp * kGS;
  a.cap_lo = n;  // code rows per unit; meta rows per unit = n / 64
  a.ngroups = ngrp;
  a.k_lo = codes;
  a.k_meta = meta;
  const dim3 grid(ngrp, units);
  if (bits == 2) channel_close_kernel<2, false><<<grid, kTileThreads, 0, s>>>(a);
  else if (bits == 4) channel_close_kernel<4, false><<<grid, kTileThreads, 0, s>>>(a);
  else channel_close_kernel<8, false><<<grid, kTileThreads, 0, s>>>(a);
  return check_launch("channel_close_kernel (keys)");
}

// Per-channel keys: the prefill's retained tokens (n_lo must be a multiple of 64): full groups
// are closed at once, the tail waits in the buffer.
int channel_append_lo(const uint16_t* k, const uint16_t* v, int src_len, const int32_t* src_pos, int n_tokens,
                      int pos_base, const mikv_cache* c, cudaStream_t s) {
  if (c->n_lo % kGS)
    return fail(MIKV_ESHAPE, "quantize_append(LO): per-channel keys append to a closed group boundary (n_lo=%d)",
                c->n_lo);
  if ((!k || !v) && n_tokens > 0) return fail(MIKV_EINVAL, "quantize_append: null k/v");
  if (n_tokens < 0 || src_len < 1) return fail(MIKV_ESHAPE, "quantize_append: n_tokens/src_len");
  if (c->n_lo + n_tokens > c->cap_lo)
    return fail(MIKV_ESHAPE, "quantize_append: tier capacity %d exceeded (%d + %d)", c->cap_lo, c->n_lo, n_tokens);
  if (!c->k_lo || !c->v_lo || !c->k_lo_meta || !c->v_lo_meta || !c->pos_lo)
    return fail(MIKV_EINVAL, "quantize_append: null tier buffer");
  if (!aligned16(c->k_lo) || !aligned16(c->v_lo) || !aligned16(c->k_lo_meta) || !aligned16(c->v_lo_meta) ||
      (k && !aligned16(k)) || (v && !aligned16(v)))
    return fail(MIKV_EALIGN, "quantize_append: buffers must be 16-byte aligned");
  if (n_tokens == 0) return MIKV_OK;
  const long units = static_cast<long>(c->B) * c->Hkv;
  if (units > 65535) return fail(MIKV_ESHAPE, "quantize_append: B*Hkv=%ld above 65535", units);
  ChanArgs a = chan_args(c);
  a.k = reinterpret_cast<const __half*>(k);
  a.v = reinterpret_cast<const __half*>(v);
  a.src_pos = src_pos;
  a.src_stride = src_len;
  a.src_len = src_len;
  a.n_tokens = n_tokens;
  a.pos_base = pos_base;
  a.base_slot = c->n_lo;
  a.ngroups = n_tokens / kGS;
  const int ctas = a.ngroups + (n_tokens % kGS ? 1 : 0);
  return launch_close(a, dim3(ctas, static_cast<unsigned>(units)), c->lo_bits, s);
}

// Per-channel keys: close the group whose 64 pairs wait in the buffer (c->n_lo is the count
// with the 64th pair included, a multiple of 64).
int channel_close_waiting(const mikv_cache* c, cudaStream_t s) {
  ChanArgs a = chan_args(c);
  a.k = static_cast<const __half*>(c->k_pend);
  a.v = static_cast<const __half*>(c->v_pend);
  a.src_stride = kGS;
  a.src_len = kGS;
  a.n_tokens = kGS;
  a.base_slot = c->n_lo - kGS;
  a.ngroups = 1;
  return launch_close(a, dim3(1, static_cast<unsigned>(c->B * c->Hkv)), c->lo_bits, s);
}

}  // namespace mikv

extern "C" int mikv_quantize_append(int tier, const uint16_t* k, const uint16_t* v, int src_len,
                                    const int32_t* src_pos, int n_tokens, int pos_base,
                                    const float* src_scores, mikv_cache* c, void* stream) {
  clear_error();
  if (int e = validate_cache(c, "quantize_append")) return e;
  if (!src_pos && n_tokens > 0) return fail(MIKV_EINVAL, "quantize_append: null src_pos");
  cudaStream_t s = as_stream(stream);
  if (tier == MIKV_TIER_HI || tier == MIKV_TIER_LO) {
    const bool hi = tier == MIKV_TIER_HI;
    if (!hi && c->key_mode == MIKV_KEYS_PER_CHANNEL) {
      if (int e = channel_append_lo(k, v, src_len, src_pos, n_tokens, pos_base, c, s)) return e;
    } else if (int e = append_tokens(hi, k, v, src_len, src_pos, n_tokens, pos_base, src_scores, c, s)) {
      return e;
    }
    if (hi) c->n_hi += n_tokens;
    else c->n_lo += n_tokens;
    return MIKV_OK;
  }
  if (tier == MIKV_TIER_DEMOTE) {
    if (n_tokens != 1) return fail(MIKV_ESHAPE, "quantize_append(DEMOTE): n_tokens must be 1");
    DemoteArgs a;
    if (int e = demote_args(c, src_pos, a)) return e;
    const long units = static_cast<long>(c->B) * c->Hkv;
    demote_kernel<<<static_cast<unsigned>((units + 7) / 8), 256, 0, s>>>(a);
    if (int e = check_launch("demote_kernel")) return e;
    c->n_hi -= 1;
    c->n_lo += 1;
    // per-channel keys: the 64th waiting pair closes its group
    if (c->key_mode == MIKV_KEYS_PER_CHANNEL && c->n_lo % kGS == 0) return channel_close_waiting(c, s);
    return MIKV_OK;
  }
  return fail(MIKV_EINVAL, "quantize_append: bad tier %d", tier);
}
