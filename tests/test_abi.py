"""C ABI checks that need no GPU: the library loads, exports every call the header
declares, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mikv.h")


@pytest.fixture(scope="session")
def lib():
    from mixed_precision_kv_balancer_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build_library()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(mikv_\w+)\s*\(", src, re.M)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("mikv_balance_prefill", "mikv_quantize_append", "mikv_score_update", "mikv_select",
              "mikv_decode_attention", "mikv_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from mixed_precision_kv_balancer_gb300 import _lib
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(_lib.EXPORTS)


def _cache(**kw):
    from mixed_precision_kv_balancer_gb300 import _lib
    c = _lib.mikv_cache()
    c.B, c.Hkv, c.Hq, c.D, c.hi_bits, c.lo_bits = 1, 2, 4, 128, 16, 2
    c.cap_hi, c.cap_lo, c.n_hi, c.n_lo = 8, 8, 0, 0
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_workspace_queries(lib):
    assert lib.mikv_balance_workspace_bytes(2, 4, 128) == 2 * 2 * 4 * 128 * 4
    assert lib.mikv_score_workspace_bytes(1, 4, 100) >= 4 * 100 * 4
    assert lib.mikv_select_workspace_bytes(0, 1, 8, 40, 1000, 5120) == 0      # H2O needs none
    assert lib.mikv_select_workspace_bytes(1, 1, 8, 40, 1000, 5120) >= 8 * 1000 * 4
    # operand tiles (32 KB per head and 32-row batch block) + per-column partial sums
    assert lib.mikv_output_perturbation_workspace_bytes(64, 32, 4096) >= 32 * 2 * 32768 + 64 * 32 * 128 * 4
    assert lib.mikv_output_perturbation_workspace_bytes(1, 40, 5120) >= 40 * 32768 + 40 * 160 * 4
    assert lib.mikv_output_perturbation_workspace_bytes(1, 4, 32) == 0        # hidden below one column block
    c = _cache(cap_hi=1000, cap_lo=4000)
    assert lib.mikv_decode_workspace_bytes(ctypes.byref(c)) > 0
    bad = _cache(D=64)
    assert lib.mikv_decode_workspace_bytes(ctypes.byref(bad)) == 0


def test_host_side_rejections(lib):
    """Every rejection happens before a launch (this process has no GPU)."""
    EINVAL, ESHAPE, EALIGN, EUNSUP = -1, -2, -3, -4
    fake = ctypes.c_void_p(4096)
    assert lib.mikv_balance_prefill(None, None, 1, 4, 2, 8, 128, None, None, 0, None) == EINVAL
    assert lib.mikv_balance_prefill(fake, fake, 1, 4, 2, 8, 64, fake, fake, 1 << 20, None) == EUNSUP
    assert lib.mikv_balance_prefill(fake, fake, 1, 3, 2, 8, 128, fake, fake, 1 << 20, None) == ESHAPE
    assert lib.mikv_balance_prefill(ctypes.c_void_p(4098), fake, 1, 4, 2, 8, 128, fake, fake, 1 << 20, None) == EALIGN
    assert lib.mikv_balance_prefill(fake, fake, 1, 4, 2, 8, 128, fake, fake, 16, None) == ESHAPE
    assert b"workspace" in lib.mikv_last_error()
    c = _cache()
    assert lib.mikv_quantize_append(7, fake, fake, 8, fake, 1, 0, None, ctypes.byref(c), None) == EINVAL
    c = _cache(lo_bits=3)
    assert lib.mikv_quantize_append(1, fake, fake, 8, fake, 1, 0, None, ctypes.byref(c), None) == EUNSUP
    c = _cache(n_lo=8)
    c.k_lo = c.v_lo = c.k_lo_meta = c.v_lo_meta = c.pos_lo = 4096
    assert lib.mikv_quantize_append(1, fake, fake, 8, fake, 1, 0, None, ctypes.byref(c), None) == ESHAPE
    assert b"capacity" in lib.mikv_last_error()
    c = _cache()
    assert lib.mikv_decode_attention(fake, ctypes.byref(c), fake, fake, None, fake, 1 << 20, None) == ESHAPE
    c = _cache(n_hi=9)
    assert lib.mikv_decode_attention(fake, ctypes.byref(c), fake, fake, None, fake, 1 << 20, None) == ESHAPE
    c = _cache()
    assert lib.mikv_select(5, ctypes.byref(c), 10, 20, 2, 0.5, fake, None, None, None, 0, None,
                           fake, fake, None, None, 0, None) == EINVAL
    assert lib.mikv_select(1, ctypes.byref(c), 10, 20, 2, 1.5, fake, fake, None, None, 0, fake,
                           fake, fake, None, fake, 1 << 20, None) == EINVAL
    assert lib.mikv_select(0, ctypes.byref(c), 10, 120, 2, 0.5, fake, None, None, None, 0, None,
                           fake, fake, None, None, 0, None) == ESHAPE
    c = _cache(n_hi=2, cap_hi=8)
    c.scores = c.pos_hi = 4096
    assert lib.mikv_select(2, ctypes.byref(c), 10, 20, 4, 0.5, None, None, None, None, 0, None,
                           None, fake, None, None, 0, None) == ESHAPE     # n_hi <= window
    assert lib.mikv_score_update(9, None, None, 0, None, None, ctypes.byref(_cache()), None, None,
                                 None, 0, None) == EINVAL
    # the step after attention
    op = lib.mikv_output_perturbation
    assert op(None, None, None, 1, 4, 128, 128, None, fake, None, 0, None) == EINVAL      # null o
    assert op(fake, None, fake, 1, 4, 128, 128, None, fake, fake, 1 << 20, None) == EINVAL  # pert needs o_hat
    assert op(fake, fake, None, 1, 4, 128, 128, fake, None, None, 0, None) == EINVAL      # y needs w_o_t
    assert op(fake, fake, fake, 1, 4, 64, 128, fake, fake, fake, 1 << 20, None) == EUNSUP
    assert op(fake, fake, fake, 0, 4, 128, 128, fake, fake, fake, 1 << 20, None) == ESHAPE
    assert op(fake, fake, fake, 1, 4, 128, 192, fake, fake, fake, 1 << 20, None) == ESHAPE  # hidden % 128
    assert op(fake, fake, fake, 1, 4, 128, 128, fake, fake, fake, 64, None) == ESHAPE      # workspace
    assert op(fake, fake, ctypes.c_void_p(4098), 1, 4, 128, 128, fake, fake, fake, 1 << 20, None) == EALIGN
    assert op(fake, fake, fake, 1, 4, 128, 128, None, None, None, 0, None) == 0            # nothing asked
    # post-attention top-k needs the full FP16 cache
    tk = lib.mikv_topk_attention
    c = _cache(n_hi=4)
    assert tk(None, ctypes.byref(c), 20, fake, None, None, fake, 1 << 20, None) == EINVAL
    assert tk(fake, ctypes.byref(_cache(n_hi=4, n_lo=2)), 20, fake, None, None, fake, 1 << 20, None) == EUNSUP
    assert tk(fake, ctypes.byref(_cache(n_hi=4, hi_bits=8)), 20, fake, None, None, fake, 1 << 20, None) == EUNSUP
    assert tk(fake, ctypes.byref(c), 101, fake, None, None, fake, 1 << 20, None) == ESHAPE
    assert tk(fake, ctypes.byref(_cache()), 20, fake, None, None, fake, 1 << 20, None) == ESHAPE   # n_hi 0
    assert tk(fake, ctypes.byref(c), 20, fake, None, None, fake, 16, None) == ESHAPE             # workspace
    assert lib.mikv_topk_attention_workspace_bytes(ctypes.byref(c), 20) > 0
    assert lib.mikv_topk_attention_workspace_bytes(ctypes.byref(_cache()), 20) == 0
    # per-channel group quantisation
    cqz = lib.mikv_channel_quantize
    assert cqz(None, 1, 64, 128, 2, fake, fake, None) == EINVAL
    assert cqz(fake, 1, 64, 64, 2, fake, fake, None) == EUNSUP
    assert cqz(fake, 1, 64, 128, 3, fake, fake, None) == EUNSUP
    assert cqz(fake, 0, 64, 128, 2, fake, fake, None) == ESHAPE
    assert cqz(fake, 1, 63, 128, 2, fake, fake, None) == 0          # no full group: nothing to do
    # the attention timing hook takes both events or neither
    assert lib.mikv_set_attention_events(fake, None) == EINVAL
    assert lib.mikv_set_attention_events(None, fake) == EINVAL
    assert lib.mikv_set_attention_events(None, None) == 0
    # the wait-status query needs somewhere to write
    assert lib.mikv_wait_status(None, 0) == EINVAL
    # the wait probe's poll count is bounded on the host
    assert lib.mikv_wait_probe(0, 0, None) == EINVAL
    assert lib.mikv_wait_probe((1 << 24) + 1, 0, None) == EINVAL


def test_per_channel_key_mode_rejections(lib):
    """Per-channel keys: only FP16 important tiers over INT2 / INT4, whole groups of capacity,
    waiting-pair buffers present, LO appends on a group boundary; all rejected on the host."""
    EINVAL, ESHAPE, EUNSUP = -1, -2, -4
    fake = ctypes.c_void_p(4096)

    def cache(**kw):
        c = _cache(**{"key_mode": 1, "cap_lo": 128, **kw})
        c.k_lo = c.v_lo = c.k_lo_meta = c.v_lo_meta = c.pos_lo = 4096
        if "k_pend" not in kw:
            c.k_pend = c.v_pend = 4096
        return c

    app = lambda c, n=1: lib.mikv_quantize_append(1, fake, fake, 8, fake, n, 0, None, ctypes.byref(c), None)
    assert app(_cache(key_mode=7)) == EINVAL
    assert app(cache(hi_bits=8)) == EUNSUP
    assert app(cache(lo_bits=8)) == EUNSUP
    assert app(cache(cap_lo=100)) == ESHAPE
    c = cache(k_pend=None)
    c.k_pend = c.v_pend = None
    assert app(c) == EINVAL
    assert app(cache(n_lo=10)) == ESHAPE                         # off a group boundary
    assert b"group boundary" in lib.mikv_last_error()
    assert lib.mikv_decode_workspace_bytes(ctypes.byref(cache(cap_hi=64))) > \
        lib.mikv_decode_workspace_bytes(ctypes.byref(_cache(cap_hi=64, cap_lo=128)))
