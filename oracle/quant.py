"""Per-token asymmetric group quantizer and bit packing (oracle).

Sources:
* MiKV reading notes (velog), "Key contributions, 1)": evicted KV pairs are
  kept with plain per-token asymmetric quantisation (the LLM-QAT scheme).
* Same notes, "2) Outlier-aware handling", supplementary remarks: the group
  size is half the attention head dimension (mitigates RoPE artefacts); keys
  are quantised as I(k * b) with the channel balancer b.
* paperlayer summary of arXiv 2402.18096v1, Appendix C: per-token quantisation
  was adopted.

Arithmetic (float32, round-to-nearest-even for every operation, in this order;
the pages fix none of it, so this is the stated reading):

  x      : the group's values as float32 (keys: fl(k * b); values: v)
  mn, mx : exact minimum and maximum of the group
  s32    = fl( fl(mx - mn) / qmax ),  qmax = 2**bits - 1
  s      = half(s32),  z = half(mn)                (stored as an fp16 pair)
  code   = clamp( rint_even( fl( fl(x - float(z)) / float(s) ) ), 0, qmax )
           and code = 0 for every element when float(s) == 0
  dequant: x~ = float(s) * code + float(z)

The zero point is the fp16 group minimum (a float offset), not an integer.

Packing: channel c of a token row takes bits [(c*bits) mod 8, +bits) of byte
floor(c*bits/8), least significant bits first.  A row is D*bits/8 bytes.
Meta: per group the pair (scale, zero) as two consecutive binary16 values.
"""
import numpy as np

QMAX = {2: 3, 4: 15, 8: 255}


def balance_keys(k: np.ndarray, b: np.ndarray | None) -> np.ndarray:
    """fl32(k * b) channel-wise; k fp16 [..., D], b float32 broadcastable [..., D] or None."""
    x = k.astype(np.float32)
    if b is None:
        return x
    return (x * b.astype(np.float32)).astype(np.float32)


def quantize_groups(x: np.ndarray, bits: int, gs: int):
    """x float32 [..., D] -> (codes uint8 [..., D], meta uint16 [..., D//gs, 2] = fp16 bits of (scale, zero))."""
    assert x.dtype == np.float32 and bits in QMAX
    D = x.shape[-1]
    assert D % gs == 0
    qmax = np.float32(QMAX[bits])
    xg = x.reshape(*x.shape[:-1], D // gs, gs)
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    s32 = ((mx - mn).astype(np.float32) / qmax).astype(np.float32)
    s = s32.astype(np.float16)
    z = mn.astype(np.float16)
    sf = s.astype(np.float32)[..., None]
    zf = z.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xg - zf).astype(np.float32) / sf).astype(np.float32)
    codes = np.clip(np.rint(t), 0, qmax)
    codes = np.where(sf == 0, 0, codes)
    codes = codes.astype(np.uint8).reshape(x.shape)
    meta = np.stack([s.view(np.uint16), z.view(np.uint16)], axis=-1)
    return codes, meta


def dequantize(codes: np.ndarray, meta: np.ndarray, gs: int) -> np.ndarray:
    """Exact dequantisation s*code + z in float64 (all three are exact in float64)."""
    D = codes.shape[-1]
    s = meta[..., 0].view(np.float16).astype(np.float64)[..., None]
    z = meta[..., 1].view(np.float16).astype(np.float64)[..., None]
    c = codes.astype(np.float64).reshape(*codes.shape[:-1], D // gs, gs)
    return (s * c + z).reshape(codes.shape)


def dequantize_f32(codes: np.ndarray, meta: np.ndarray, gs: int) -> np.ndarray:
    """float32 dequantisation fl(fl(s*code) + z), the value re-quantised when an INT8 slot is demoted."""
    D = codes.shape[-1]
    s = meta[..., 0].view(np.float16).astype(np.float32)[..., None]
    z = meta[..., 1].view(np.float16).astype(np.float32)[..., None]
    c = codes.astype(np.float32).reshape(*codes.shape[:-1], D // gs, gs)
    prod = (s * c).astype(np.float32)
    return (prod + z).astype(np.float32).reshape(codes.shape)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes uint8 [..., D] (each < 2**bits) -> packed uint8 [..., D*bits//8]."""
    if bits == 8:
        return codes.astype(np.uint8).copy()
    per = 8 // bits
    D = codes.shape[-1]
    c = codes.astype(np.uint32).reshape(*codes.shape[:-1], D // per, per)
    shifts = (np.arange(per, dtype=np.uint32) * bits)
    return (c << shifts).sum(axis=-1).astype(np.uint8)


def unpack_codes(packed: np.ndarray, bits: int, D: int) -> np.ndarray:
    """Inverse of pack_codes."""
    if bits == 8:
        return packed.astype(np.uint8).copy()
    per = 8 // bits
    p = packed.astype(np.uint32)[..., None]
    shifts = (np.arange(per, dtype=np.uint32) * bits)
    c = (p >> shifts) & ((1 << bits) - 1)
    return c.reshape(*packed.shape[:-1], D).astype(np.uint8)
