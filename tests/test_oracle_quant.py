"""Pins for the oracle's per-token asymmetric quantizer and bit packing (no GPU).

Definition: MiKV reading notes (velog), "Key contributions, 1)" (per-token
asymmetric quantisation, LLM-QAT) and "2)" supplementary remarks (group size =
half the head dimension; keys quantised as I(k*b)).
"""
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import quant


def _load_hand():
    rows = []
    with open(os.path.join(GOLDEN, "quant_hand.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, x, s, z, codes = [p.strip() for p in line.split("|")]
            rows.append((int(bits), [float(v) for v in x.split()], float(s), float(z),
                         [int(c) for c in codes.split()]))
    return rows


@pytest.mark.parametrize("row", _load_hand())
def test_hand_cases(row):
    bits, x, s, z, codes = row
    c, meta = quant.quantize_groups(np.array(x, np.float32)[None, :], bits, 4)
    np.testing.assert_array_equal(c[0], codes)
    assert meta[0, 0, 0].view(np.float16) == np.float16(s)
    assert meta[0, 0, 1].view(np.float16) == np.float16(z)


def _groups(rng, n, gs=64):
    x = rng.standard_normal((n, gs)).astype(np.float32)
    x[::3] *= 16                       # outlier-scale groups
    x[1::7, 5] = 40.0                  # a single outlier inside a group
    return x


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_are_nearest_level(bits):
    """Brute force: each code is the nearest of the 2**bits levels s*j + z (exact arithmetic),
    except within float32 rounding of a midpoint, where either neighbour is accepted."""
    rng = np.random.default_rng(bits)
    x = _groups(rng, 400)
    codes, meta = quant.quantize_groups(x, bits, 64)
    s = meta[:, 0, 0].view(np.float16).astype(np.float64)
    z = meta[:, 0, 1].view(np.float16).astype(np.float64)
    qmax = 2 ** bits - 1
    levels = s[:, None] * np.arange(qmax + 1)[None, :] + z[:, None]          # [n, L]
    dist = np.abs(x.astype(np.float64)[:, :, None] - levels[:, None, :])    # [n, gs, L]
    best = dist.argmin(axis=2)
    t = (x.astype(np.float64) - z[:, None]) / s[:, None]
    near_mid = np.abs(np.abs(t - np.floor(t)) - 0.5) < 1e-5 * np.maximum(1, np.abs(t))
    ok = (codes == best) | (near_mid & (np.abs(codes.astype(int) - best) <= 1))
    assert ok.all()


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound(bits):
    """|x - x~| <= s/2 + |mn - z| + qmax*|s32 - s| (+ float32 slack) for every element."""
    rng = np.random.default_rng(10 + bits)
    x = _groups(rng, 500)
    codes, meta = quant.quantize_groups(x, bits, 64)
    xt = quant.dequantize(codes, meta, 64)
    qmax = 2 ** bits - 1
    mn = x.min(axis=1).astype(np.float64)
    s32 = (x.max(axis=1).astype(np.float64) - mn) / qmax
    s = meta[:, 0, 0].view(np.float16).astype(np.float64)
    z = meta[:, 0, 1].view(np.float16).astype(np.float64)
    bound = s / 2 + np.abs(mn - z) + qmax * np.abs(s32 - s)
    err = np.abs(x.astype(np.float64) - xt).max(axis=1)
    assert (err <= bound * (1 + 1e-6) + 1e-7).all()


def test_constant_group_and_exact_grid():
    x = np.full((1, 64), 3.25, np.float32)
    codes, meta = quant.quantize_groups(x, 2, 64)
    assert (codes == 0).all()
    assert quant.dequantize(codes, meta, 64)[0, 0] == 3.25
    # values on the grid mn + j*s with s a power of two reconstruct exactly
    j = np.tile(np.arange(16), 4)
    x = (-1.5 + j * 0.125).astype(np.float32)[None, :]
    codes, meta = quant.quantize_groups(x, 4, 64)
    np.testing.assert_array_equal(codes[0], j)
    np.testing.assert_array_equal(quant.dequantize(codes, meta, 64)[0], x[0].astype(np.float64))


def test_groups_are_independent_halves():
    """Group size 64 on D=128: the two halves of a row get their own (scale, zero)."""
    x = np.concatenate([np.linspace(0, 3, 64), np.linspace(-100, 100, 64)]).astype(np.float32)[None]
    codes, meta = quant.quantize_groups(x, 2, 64)
    assert meta.shape == (1, 2, 2)
    assert meta[0, 0, 1].view(np.float16) == 0 and meta[0, 1, 1].view(np.float16) == -100
    assert meta[0, 0, 0].view(np.float16) == 1


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_layout_bitwise(bits):
    """Channel c occupies bits [(c*bits) % 8, +bits) of byte (c*bits)//8, LSB first (np.unpackbits)."""
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(5, 128)).astype(np.uint8)
    packed = quant.pack_codes(codes, bits)
    assert packed.shape == (5, 128 * bits // 8)
    bitstream = np.unpackbits(packed, axis=1, bitorder="little")          # [5, 128*bits]
    for c in range(128):
        val = np.zeros(5, np.int64)
        for j in range(bits):
            val |= bitstream[:, c * bits + j].astype(np.int64) << j
        np.testing.assert_array_equal(val, codes[:, c])
    np.testing.assert_array_equal(quant.unpack_codes(packed, bits, 128), codes)


def test_balanced_keys_are_float32_products():
    k = np.array([[1.5, -2.0, 3.0]], np.float16)
    b = np.array([1.0 / 3.0, 2.0, 0.1], np.float32)
    x = quant.balance_keys(k, b)
    assert x.dtype == np.float32
    np.testing.assert_array_equal(x, np.float32(k.astype(np.float32) * b))
    assert x[0, 1] == -4.0


def test_dequantize_f32_order():
    """fl32(s * code + z), rounded once to float32, against bit patterns derived by hand.

    s = fp16 0x3C01 = 1025/1024, z = fp16 0x8401 = -(1025/1024) * 2^-14, code 255:
    s*code = 261375/1024 = 255.2490234375 (exact: 19 significant bits), and
    s*code + z = 255.24896234273910522...; float32 spacing at 2^7 is 2^-16, and the sum is
    16727995 + 255/256 spacings, so it rounds up to 16727996 * 2^-16 = 255.24896240234375,
    bits 0x437F3FBC.
    s = 0x3C01, z = fp16 0x0001 = 2^-24, code 3: 3075/1024 + 2^-24 = 3.00292974710464...;
    spacing at 2^1 is 2^-22, the sum is 12595200 + 1/4 spacings, rounds down to
    3.0029296875, bits 0x40403000."""
    def one(s_bits, z_bits, code):
        meta = np.array([[[s_bits, z_bits]]], np.uint16)
        codes = np.full((1, 4), code, np.uint8)
        got = quant.dequantize_f32(codes, meta, 4)
        assert got.dtype == np.float32
        return got[0].view(np.uint32)
    np.testing.assert_array_equal(one(0x3C01, 0x8401, 255), np.full(4, 0x437F3FBC, np.uint32))
    np.testing.assert_array_equal(one(0x3C01, 0x0001, 3), np.full(4, 0x40403000, np.uint32))
