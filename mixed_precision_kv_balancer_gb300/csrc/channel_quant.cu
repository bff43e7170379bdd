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
namespace {

constexpr int kCqGroup = 64;

// One CTA per (group, unit), one thread per channel.
__global__ void __launch_bounds__(kD) channel_group_quant_kernel(const __half* __restrict__ k, int n, int bits,
                                                                 uint8_t* __restrict__ codes,
                                                                 __half2* __restrict__ meta) {
  __shared__ uint8_t cs[kCqGroup][kD];
  const int grp = blockIdx.x, ngrp = gridDim.x;
  const long unit = blockIdx.y;
  const int c = threadIdx.x;
  const __half* src = k + (unit * n + static_cast<long>(grp) * kCqGroup) * kD + c;
  float x[kCqGroup];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int t = 0; t < kCqGroup; ++t) {
    x[t] = __half2float(src[static_cast<long>(t) * kD]);
    mn = fminf(mn, x[t]);
    mx = fmaxf(mx, x[t]);
  }
  const int qmax = (1 << bits) - 1;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(qmax));
  const __half sh = __float2half_rn(s32), zh = __float2half_rn(mn);
  const float sf = __half2float(sh), zf = __half2float(zh);
  meta[(unit * ngrp + grp) * kD + c] = __halves2half2(sh, zh);
#pragma unroll
  for (int t = 0; t < kCqGroup; ++t) {
    int q = 0;
    if (sf != 0.f) q = min(max(__float2int_rn(__fdiv_rn(__fsub_rn(x[t], zf), sf)), 0), qmax);
    cs[t][c] = static_cast<uint8_t>(q);
  }
  __syncthreads();
  // pack: row t holds kD * bits / 8 bytes; byte j carries channels j*per .. j*per + per - 1
  const int per = 8 / bits, row_bytes = kD * bits / 8;
  uint8_t* dst = codes + (unit * n + static_cast<long>(grp) * kCqGroup) * row_bytes;
  for (int i = threadIdx.x; i < kCqGroup * row_bytes; i += kD) {
    const int t = i / row_bytes, j = i % row_bytes;
    uint32_t byte = 0;
    for (int e = 0; e < per; ++e) byte |= static_cast<uint32_t>(cs[t][j * per + e]) << (e * bits);
    dst[static_cast<long>(t) * row_bytes + j] = static_cast<uint8_t>(byte);
  }
}

}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" int mikv_channel_quantize(const uint16_t* k, int units, int n, int D, int bits, uint8_t* codes,
                                     uint16_t* meta, void* stream) {
  clear_error();
  if (!k || !codes || !meta) return fail(MIKV_EINVAL, "channel_quantize: null pointer");
  if (D != kD) return fail(MIKV_EUNSUPPORTED, "channel_quantize: D=%d (only %d)", D, kD);
  if (bits != 2 && bits != 4 && bits != 8) return fail(MIKV_EUNSUPPORTED, "channel_quantize: bits=%d", bits);
  if (units < 1 || n < 0 || units > 65535) return fail(MIKV_ESHAPE, "channel_quantize: units=%d n=%d", units, n);
  const int ngrp = n / kCqGroup;
  if (ngrp == 0) return MIKV_OK;  // every key is still pending
  channel_group_quant_kernel<<<dim3(ngrp, units), kD, 0, as_stream(stream)>>>(
      reinterpret_cast<const __half*>(k), n, bits, codes, reinterpret_cast<__half2*>(meta));
  return check_launch("channel_group_quant_kernel");
}
