// Per-channel group quantisation of retained-tier keys: the first stage of the per-channel
// key alternative (MiKV reading notes, Appendix C remarks; paperlayer summary, "C.
// Experiments on per-channel quantization of keys": group size 64, keys per channel).
// Reading: a group is 64 consecutive keys of one (batch, key head); per channel c the group's
// 64 values are quantised with the per-token quantizer's arithmetic along the token axis:
// s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn), code = clamp(rint_even(fl(fl(x - z) / s)),
// 0, qmax), 0 where s == 0.  Codes are stored in the per-token rows of the low tier (channel c
// at bits (c*bits) mod 8 of byte c*bits/8, LSB first); meta per (group, channel).
#include "common.cuh"

namespace mikv {
// In quantize.cu: the same group-closing kernel the per-channel cache uses, keys only (one CTA
// per (group, unit): the group's 64 rows staged in shared memory with 16-byte copies, one
// thread per channel, codes packed per row with 16-byte stores).
int channel_quantize_keys(const __half* k, int units, int n, int bits, uint8_t* codes, __half2* meta,
                          cudaStream_t s);
}  // namespace mikv

using namespace mikv;

extern "C" int mikv_channel_quantize(const uint16_t* k, int units, int n, int D, int bits, uint8_t* codes,
                                     uint16_t* meta, void* stream) {
  clear_error();
  if (!k || !codes || !meta) return fail(MIKV_EINVAL, "channel_quantize: null pointer");
  if (D != kD) return fail(MIKV_EUNSUPPORTED, "channel_quantize: D=%d (only %d)", D, kD);
  if (bits != 2 && bits != 4 && bits != 8) return fail(MIKV_EUNSUPPORTED, "channel_quantize: bits=%d", bits);
  if (units < 1 || n < 0 || units > 65535) return fail(MIKV_ESHAPE, "channel_quantize: units=%d n=%d", units, n);
  if (!aligned16(k) || !aligned16(codes) || !aligned16(meta))
    return fail(MIKV_EALIGN, "channel_quantize: k, codes and meta must be 16-byte aligned");
  return channel_quantize_keys(reinterpret_cast<const __half*>(k), units, n, bits, codes,
                               reinterpret_cast<__half2*>(meta), as_stream(stream));
}
