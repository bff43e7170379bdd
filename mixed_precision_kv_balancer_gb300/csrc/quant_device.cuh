// Device routines shared by the quantise/append, demotion and fused decode-step kernels
// (internal; not part of the C ABI).  Quantisation arithmetic, in this order, with
// round-to-nearest intrinsics:  x = fl(k*b) for keys of a quantised tier or v;
// s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn);
// code = clamp(rint_even(fl(fl(x - z) / s)), 0, qmax), 0 where s == 0.
#pragma once
#include "common.cuh"

namespace mikv {

struct Row4 {
  float x[4];
};

__device__ __forceinline__ Row4 load_fp16x4(const __half* p) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __half2 a = *reinterpret_cast<__half2*>(&u.x), b = *reinterpret_cast<__half2*>(&u.y);
  Row4 r;
  r.x[0] = __low2float(a);
  r.x[1] = __high2float(a);
  r.x[2] = __low2float(b);
  r.x[3] = __high2float(b);
  return r;
}

// Quantise the 4 channels this lane owns (its half-warp is one group); returns the
// codes packed LSB-first in a 32-bit word (bits*4 significant bits) and the meta pair.
__device__ __forceinline__ uint32_t quantize4(const Row4& r, int bits, uint32_t& meta) {
  float mn = fminf(fminf(r.x[0], r.x[1]), fminf(r.x[2], r.x[3]));
  float mx = fmaxf(fmaxf(r.x[0], r.x[1]), fmaxf(r.x[2], r.x[3]));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const int qmax = (1 << bits) - 1;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(qmax));
  const __half sh = __float2half_rn(s32), zh = __float2half_rn(mn);
  const float sf = __half2float(sh), zf = __half2float(zh);
  meta = pack_half2(sh, zh);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int c = 0;
    if (sf != 0.f) {
      c = __float2int_rn(__fdiv_rn(__fsub_rn(r.x[i], zf), sf));
      c = min(max(c, 0), qmax);
    }
    packed |= static_cast<uint32_t>(c) << (i * bits);
  }
  return packed;
}

__device__ __forceinline__ void store_codes(uint8_t* row, int lane, int bits, uint32_t packed) {
  if (bits == 2) row[lane] = static_cast<uint8_t>(packed);
  else if (bits == 4) reinterpret_cast<uint16_t*>(row)[lane] = static_cast<uint16_t>(packed);
  else reinterpret_cast<uint32_t*>(row)[lane] = packed;
}

__device__ __forceinline__ void store_meta(__half2* meta_row, int lane, uint32_t meta) {
  if ((lane & 15) == 0) reinterpret_cast<uint32_t*>(meta_row)[lane >> 4] = meta;
}

struct DemoteArgs {
  const int32_t* victim;  // [B*Hkv]
  const float* bal;
  int units, hi_bits, lo_bits, cap_hi, cap_lo, n_hi, n_lo;
  int key_mode;           // MIKV_KEYS_PER_CHANNEL: the pair joins the waiting buffer
  __half *k_pend, *v_pend;  // [B*Hkv][64][D]
  uint8_t *k_hi, *v_hi;
  __half2 *k_hi_meta, *v_hi_meta;
  uint8_t *k_lo, *v_lo;
  __half2 *k_lo_meta, *v_lo_meta;
  int32_t *pos_hi, *pos_lo;
  float* scores;
};

// The 4 channels 4*lane.. of a 4-bit code row, dequantised as fl(fl(s*code) + z).
__device__ __forceinline__ Row4 dequant_int4x4(const uint8_t* row, const __half2* meta, int lane) {
  const uint32_t w = reinterpret_cast<const uint16_t*>(row)[lane];
  const __half2 m = meta[lane >> 4];
  const float sf = __low2float(m), zf = __high2float(m);
  Row4 r;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    r.x[i] = __fadd_rn(__fmul_rn(sf, static_cast<float>((w >> (4 * i)) & 0xfu)), zf);
  return r;
}

__device__ __forceinline__ Row4 dequant_int8x4(const uint8_t* row, const __half2* meta, int lane) {
  const uint32_t w = reinterpret_cast<const uint32_t*>(row)[lane];
  const __half2 m = meta[lane >> 4];
  const float sf = __low2float(m), zf = __high2float(m);
  Row4 r;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    r.x[i] = __fadd_rn(__fmul_rn(sf, static_cast<float>((w >> (8 * i)) & 0xffu)), zf);
  return r;
}

// Move important slot `vslot` of `unit` into the low tier (re-quantised) and the last
// important slot into its place.  One warp; lanes own 4 channels each.  The last slot's
// contents are loaded first: they do not depend on the victim, so both loads overlap.
__device__ __forceinline__ void demote_one(const DemoteArgs& a, long unit, int vslot, int lane) {
  if (vslot < 0 || vslot >= a.n_hi) return;  // invalid victim: nothing moves
  const long hs = unit * a.cap_hi + vslot;
  const long last = unit * a.cap_hi + (a.n_hi - 1);
  const long ls = unit * a.cap_lo + a.n_lo;
  const bool move = hs != last;
  const int hrb = kD * a.hi_bits / 8;  // bytes per important row
  const int words = hrb / 4;           // 64, 32 or 16: lane owns words lane, lane + 32
  uint32_t lk0 = 0, lk1 = 0, lv0 = 0, lv1 = 0;
  __half2 lkm = {}, lvm = {};
  int lpos = 0;
  float lsc = 0.f;
  if (move) {
    const uint32_t* sk = reinterpret_cast<const uint32_t*>(a.k_hi + last * hrb);
    const uint32_t* sv = reinterpret_cast<const uint32_t*>(a.v_hi + last * hrb);
    if (lane < words) {
      lk0 = sk[lane];
      lv0 = sv[lane];
    }
    if (words > 32) {
      lk1 = sk[lane + 32];
      lv1 = sv[lane + 32];
    }
    if (a.hi_bits != 16 && lane < 2) {
      lkm = a.k_hi_meta[last * 2 + lane];
      lvm = a.v_hi_meta[last * 2 + lane];
    }
    if (lane == 0) {
      lpos = a.pos_hi[last];
      lsc = __ldcg(a.scores + last);  // may have been updated by another CTA
    }
  }
  if (a.key_mode == MIKV_KEYS_PER_CHANNEL) {
    // per-channel keys (FP16 important tier): the pair waits unquantised in row n_lo % 64 of
    // the buffer; the group is closed by a separate launch once 64 pairs wait
    const long pr = unit * kGS + (a.n_lo & (kGS - 1));
    reinterpret_cast<uint2*>(a.k_pend + pr * kD)[lane] = reinterpret_cast<const uint2*>(a.k_hi + hs * kD * 2)[lane];
    reinterpret_cast<uint2*>(a.v_pend + pr * kD)[lane] = reinterpret_cast<const uint2*>(a.v_hi + hs * kD * 2)[lane];
    if (lane == 0) a.pos_lo[ls] = a.pos_hi[hs];
  } else {
    Row4 xk, xv;
    if (a.hi_bits == 16) {
      xk = load_fp16x4(reinterpret_cast<const __half*>(a.k_hi) + hs * kD + lane * 4);
      xv = load_fp16x4(reinterpret_cast<const __half*>(a.v_hi) + hs * kD + lane * 4);
      if (a.bal) {
        const float4 bb = *reinterpret_cast<const float4*>(a.bal + unit * kD + lane * 4);
        xk.x[0] = __fmul_rn(xk.x[0], bb.x);
        xk.x[1] = __fmul_rn(xk.x[1], bb.y);
        xk.x[2] = __fmul_rn(xk.x[2], bb.z);
        xk.x[3] = __fmul_rn(xk.x[3], bb.w);
      }
    } else if (a.hi_bits == 8) {  // quantised tiers hold balanced keys already
      xk = dequant_int8x4(a.k_hi + hs * hrb, a.k_hi_meta + hs * 2, lane);
      xv = dequant_int8x4(a.v_hi + hs * hrb, a.v_hi_meta + hs * 2, lane);
    } else {
      xk = dequant_int4x4(a.k_hi + hs * hrb, a.k_hi_meta + hs * 2, lane);
      xv = dequant_int4x4(a.v_hi + hs * hrb, a.v_hi_meta + hs * 2, lane);
    }
    const int vpos = lane == 0 ? a.pos_hi[hs] : 0;
    const int rb = kD * a.lo_bits / 8;
    uint32_t mk, mv;
    const uint32_t pk = quantize4(xk, a.lo_bits, mk);
    const uint32_t pv = quantize4(xv, a.lo_bits, mv);
    store_codes(a.k_lo + ls * rb, lane, a.lo_bits, pk);
    store_codes(a.v_lo + ls * rb, lane, a.lo_bits, pv);
    store_meta(a.k_lo_meta + ls * 2, lane, mk);
    store_meta(a.v_lo_meta + ls * 2, lane, mv);
    if (lane == 0) a.pos_lo[ls] = vpos;
  }
  __syncwarp();
  // swap-remove: the last important slot moves into the freed one
  if (move) {
    uint32_t* dk = reinterpret_cast<uint32_t*>(a.k_hi + hs * hrb);
    uint32_t* dv = reinterpret_cast<uint32_t*>(a.v_hi + hs * hrb);
    if (lane < words) {
      dk[lane] = lk0;
      dv[lane] = lv0;
    }
    if (words > 32) {
      dk[lane + 32] = lk1;
      dv[lane + 32] = lv1;
    }
    if (a.hi_bits != 16 && lane < 2) {
      a.k_hi_meta[hs * 2 + lane] = lkm;
      a.v_hi_meta[hs * 2 + lane] = lvm;
    }
    if (lane == 0) {
      a.pos_hi[hs] = lpos;
      a.scores[hs] = lsc;
    }
  }
}

// Arguments of an append of source tokens into one tier (one warp per (token, key head)).
struct AppendArgs {
  const __half* k;        // [B][Hkv][src_len][D]
  const __half* v;
  const int32_t* src_pos; // [B][Hkv][n_tokens]
  const float* src_scores;
  const float* bal;       // [B][Hkv][D] or null
  int Hkv, src_len, n_tokens, pos_base;
  int cap, base_slot, bits;  // destination tier
  uint8_t* dk;            // codes [unit][cap][RB] or fp16 rows
  uint8_t* dv;
  __half2* dkm;           // [unit][cap][2]
  __half2* dvm;
  int32_t* dpos;
  float* dscores;         // hi tier only, else null
  long units_tokens;      // B*Hkv*n_tokens
  unsigned* ticket;       // [B*Hkv] cleared by token 0 of each unit, or null
};

// Append item `item` = (unit, token j) of `a`: one warp, lanes own 4 channels each.  Keys of a
// quantised tier are balanced first; the slot gets position src + pos_base and the source
// score (or 0) in the important tier.  Token 0 of each unit also clears the unit's ticket.
__device__ __forceinline__ void append_item(const AppendArgs& a, long item, int lane) {
  const long unit = item / a.n_tokens;
  const int j = static_cast<int>(item % a.n_tokens);
  if (a.ticket != nullptr && j == 0 && lane == 0) a.ticket[unit] = 0u;
  const int src = a.src_pos ? a.src_pos[item] : j;  // no list: token j of the source
  if (src < 0 || src >= a.src_len) return;  // out-of-range source: slot left unchanged
  const long slot = unit * a.cap + a.base_slot + j;
  const __half* ks = a.k + (unit * a.src_len + src) * kD + lane * 4;
  const __half* vs = a.v + (unit * a.src_len + src) * kD + lane * 4;
  if (a.bits == 16) {
    reinterpret_cast<uint2*>(a.dk + slot * kD * 2)[lane] = *reinterpret_cast<const uint2*>(ks);
    reinterpret_cast<uint2*>(a.dv + slot * kD * 2)[lane] = *reinterpret_cast<const uint2*>(vs);
  } else {
    Row4 xk = load_fp16x4(ks), xv = load_fp16x4(vs);
    if (a.bal) {
      const float4 bb = *reinterpret_cast<const float4*>(a.bal + unit * kD + lane * 4);
      xk.x[0] = __fmul_rn(xk.x[0], bb.x);
      xk.x[1] = __fmul_rn(xk.x[1], bb.y);
      xk.x[2] = __fmul_rn(xk.x[2], bb.z);
      xk.x[3] = __fmul_rn(xk.x[3], bb.w);
    }
    const int rb = kD * a.bits / 8;
    uint32_t mk, mv;
    const uint32_t pk = quantize4(xk, a.bits, mk);
    const uint32_t pv = quantize4(xv, a.bits, mv);
    store_codes(a.dk + slot * rb, lane, a.bits, pk);
    store_codes(a.dv + slot * rb, lane, a.bits, pv);
    store_meta(a.dkm + slot * 2, lane, mk);
    store_meta(a.dvm + slot * 2, lane, mv);
  }
  if (lane == 0) {
    a.dpos[slot] = src + a.pos_base;
    if (a.dscores) a.dscores[slot] = a.src_scores ? a.src_scores[item] : 0.f;
  }
}

}  // namespace mikv
