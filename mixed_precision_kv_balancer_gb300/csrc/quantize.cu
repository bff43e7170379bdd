// K2: per-token asymmetric group quantisation and append into a cache tier, and
// the demotion of one important-tier slot into the low-bit tier.
//
// Sources: "No Token Left Behind" reading notes (velog), "Key contributions 1)"
// (evicted KV kept with per-token asymmetric quantisation, LLM-QAT), "2)" (keys
// quantised as I(k*b); group size = half the head dimension), "3)" (INT8
// important tier).
//
// One warp per (token, key head): lane l owns channels 4l..4l+3, so a 64-channel
// group is one half-warp and its min/max are two 4-step shuffle reductions.  Every
// step uses explicit round-to-nearest intrinsics in the order the format fixes:
//   x = fl(k*b) (keys of a quantised tier) or v
//   s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn)
//   code = clamp(rint_even(fl(fl(x - z) / s)), 0, qmax); 0 where s == 0.
// Codes are packed LSB-first (channel c at bit c*bits of the row), meta is the
// fp16 pair (scale, zero) per group.  HBM-bound: 512 B read per token-head,
// 80/144/272/512 B written.
#include "quant_device.cuh"

namespace mikv {
namespace {

__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long item = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (item >= a.units_tokens) return;
  append_item(a, item, lane);
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

// Validate and launch an append (see append_args); after: the kernel launched just before on
// `s` is one of ours and this launch may overlap its tail.
int append_tokens(bool hi, const uint16_t* k, const uint16_t* v, int src_len, const int32_t* src_pos,
                  int n_tokens, int pos_base, const float* src_scores, const mikv_cache* c,
                  cudaStream_t s, unsigned* ticket, bool after) {
  AppendArgs a;
  if (int e = append_args(hi, k, v, src_len, src_pos, n_tokens, pos_base, src_scores, c, ticket, a))
    return e;
  if (n_tokens > 0) {
    const long blocks = (a.units_tokens + 7) / 8;
    if (after) {
      if (int e = check_launch_after(
              launch_after(append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a),
              "append_kernel"))
        return e;
    } else {
      append_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
      if (int e = check_launch("append_kernel")) return e;
    }
  }
  return MIKV_OK;
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
  if (!a.k_hi || !a.v_hi || !a.k_lo || !a.v_lo || !a.k_lo_meta || !a.v_lo_meta || !a.pos_hi ||
      !a.pos_lo || !a.scores || (c->hi_bits != 16 && (!a.k_hi_meta || !a.v_hi_meta)))
    return fail(MIKV_EINVAL, "demotion: null cache buffer");
  if (!aligned16(a.k_hi) || !aligned16(a.v_hi) || !aligned16(a.k_lo) || !aligned16(a.v_lo) ||
      !aligned16(a.k_lo_meta) || !aligned16(a.v_lo_meta))
    return fail(MIKV_EALIGN, "demotion: buffers must be 16-byte aligned");
  return MIKV_OK;
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
    if (int e = append_tokens(hi, k, v, src_len, src_pos, n_tokens, pos_base, src_scores, c, s,
                              nullptr, false))
      return e;
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
    return MIKV_OK;
  }
  return fail(MIKV_EINVAL, "quantize_append: bad tier %d", tier);
}
