"""ctypes binding of libmikv.so: the C ABI calls under the same names, taking torch tensors.

Argument marshalling only: every computation runs in the library's CUDA kernels.
There is no fallback; if the library is missing or a call fails, this raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmikv.so")

MIKV_PREFILL, MIKV_DECODE = 0, 1
MIKV_H2O, MIKV_CRITICALKV, MIKV_DEMOTE = 0, 1, 2
MIKV_TIER_HI, MIKV_TIER_LO, MIKV_TIER_DEMOTE = 0, 1, 2
MIKV_KEYS_PER_TOKEN, MIKV_KEYS_PER_CHANNEL = 0, 1

EXPORTS = (
    "mikv_balance_prefill", "mikv_balance_workspace_bytes", "mikv_balance_prefill_noalloc",
    "mikv_score_update", "mikv_score_workspace_bytes",
    "mikv_select", "mikv_select_workspace_bytes",
    "mikv_quantize_append",
    "mikv_decode_attention", "mikv_decode_workspace_bytes",
    "mikv_decode_step", "mikv_decode_step_workspace_bytes",
    "mikv_output_perturbation", "mikv_output_perturbation_workspace_bytes",
    "mikv_topk_attention", "mikv_topk_attention_workspace_bytes",
    "mikv_channel_quantize",
    "mikv_set_attention_events", "mikv_wait_status", "mikv_wait_probe", "mikv_last_error",
)


class MikvError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


class mikv_cache(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("Hq", ctypes.c_int32), ("D", ctypes.c_int32),
        ("hi_bits", ctypes.c_int32), ("lo_bits", ctypes.c_int32),
        ("cap_hi", ctypes.c_int32), ("cap_lo", ctypes.c_int32),
        ("n_hi", ctypes.c_int32), ("n_lo", ctypes.c_int32),
        ("k_hi", ctypes.c_void_p), ("v_hi", ctypes.c_void_p),
        ("k_hi_meta", ctypes.c_void_p), ("v_hi_meta", ctypes.c_void_p),
        ("k_lo", ctypes.c_void_p), ("v_lo", ctypes.c_void_p),
        ("k_lo_meta", ctypes.c_void_p), ("v_lo_meta", ctypes.c_void_p),
        ("pos_hi", ctypes.c_void_p), ("pos_lo", ctypes.c_void_p),
        ("balancer", ctypes.c_void_p), ("scores", ctypes.c_void_p),
        ("key_mode", ctypes.c_int32), ("k_pend", ctypes.c_void_p), ("v_pend", ctypes.c_void_p),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """Load libmikv.so (built in-tree by build()); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() or "
                           "python -m mixed_precision_kv_balancer_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    CP = ctypes.POINTER(mikv_cache)
    sig = {
        "mikv_balance_prefill": (I, [P, P, I, I, I, I, I, P, P, S, P]),
        "mikv_balance_workspace_bytes": (S, [I, I, I]),
        "mikv_balance_prefill_noalloc": (I, [P, P, I, I, I, I, I, P, P]),
        "mikv_score_update": (I, [I, P, P, I, P, P, CP, P, P, P, S, P]),
        "mikv_score_workspace_bytes": (S, [I, I, I]),
        "mikv_select": (I, [I, CP, I, I, I, F, P, P, P, P, I, P, P, P, P, P, S, P]),
        "mikv_select_workspace_bytes": (S, [I, I, I, I, I, I]),
        "mikv_quantize_append": (I, [I, P, P, I, P, I, I, P, CP, P]),
        "mikv_decode_attention": (I, [P, CP, P, P, P, P, S, P]),
        "mikv_decode_workspace_bytes": (S, [CP]),
        "mikv_decode_step": (I, [P, P, P, I, I, I, I, CP, P, P, P, S, P]),
        "mikv_decode_step_workspace_bytes": (S, [CP]),
        "mikv_output_perturbation": (I, [P, P, P, I, I, I, I, P, P, P, S, P]),
        "mikv_output_perturbation_workspace_bytes": (S, [I, I, I]),
        "mikv_topk_attention": (I, [P, CP, I, P, P, P, P, S, P]),
        "mikv_topk_attention_workspace_bytes": (S, [CP, I]),
        "mikv_channel_quantize": (I, [P, I, I, I, I, P, P, P]),
        "mikv_set_attention_events": (I, [P, P]),
        "mikv_wait_status": (I, [ctypes.POINTER(ctypes.c_uint), I]),
        "mikv_wait_probe": (I, [ctypes.c_int64, I, P]),
        "mikv_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors"
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(name: str, rc: int):
    if rc != 0:
        raise MikvError(name, rc, load().mikv_last_error().decode())


def _ws(nbytes: int, device, ws):
    if ws is not None:
        return ws, ws.numel() * ws.element_size()
    if nbytes == 0:
        return None, 0
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return t, nbytes


# --- the C ABI calls -----------------------------------------------------------------

def mikv_balance_prefill(q, k, b_out, ws=None, stream=None):
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    lib = load()
    w, nb = _ws(lib.mikv_balance_workspace_bytes(B, Hkv, D), q.device, ws)
    _check("mikv_balance_prefill", lib.mikv_balance_prefill(
        _ptr(q), _ptr(k), B, Hq, Hkv, T, D, _ptr(b_out), _ptr(w), nb, _stream(stream)))


def mikv_balance_prefill_noalloc(q, k, b_out, stream=None):
    """Balancer without a workspace: scratch is the library's static device array."""
    B, Hq, T, D = q.shape
    _check("mikv_balance_prefill_noalloc", load().mikv_balance_prefill_noalloc(
        _ptr(q), _ptr(k), B, Hq, k.shape[1], T, D, _ptr(b_out), _stream(stream)))


def mikv_score_update(mode, cache, q=None, k=None, T=0, hi_logits=None, lse=None,
                      scores_full=None, scores_head=None, ws=None, stream=None):
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    w, nb = None, 0
    if mode == MIKV_PREFILL:
        dev = q.device
        w, nb = _ws(lib.mikv_score_workspace_bytes(c.B, c.Hq, T), dev, ws)
    _check("mikv_score_update", lib.mikv_score_update(
        mode, _ptr(q), _ptr(k), T, _ptr(hi_logits), _ptr(lse), ctypes.byref(c),
        _ptr(scores_full), _ptr(scores_head), _ptr(w), nb, _stream(stream)))


def mikv_select(policy, cache, L, budget_pct, window, alpha=0.5, scores=None, scores_head=None,
                v=None, w_o=None, hidden=0, vwo_norm=None, keep_pos=None, evict_pos=None,
                keep_scores=None, ws=None, stream=None):
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    dev = (scores if scores is not None else evict_pos).device
    w, nb = _ws(lib.mikv_select_workspace_bytes(policy, c.B, c.Hkv, c.Hq, L, hidden), dev, ws)
    _check("mikv_select", lib.mikv_select(
        policy, ctypes.byref(c), L, budget_pct, window, float(alpha), _ptr(scores),
        _ptr(scores_head), _ptr(v), _ptr(w_o), hidden, _ptr(vwo_norm), _ptr(keep_pos),
        _ptr(evict_pos), _ptr(keep_scores), _ptr(w), nb, _stream(stream)))


def mikv_quantize_append(tier, cache, k, v, src_pos, n_tokens, pos_base=0, src_scores=None,
                         stream=None):
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    src_len = 0 if k is None else k.shape[2]
    _check("mikv_quantize_append", lib.mikv_quantize_append(
        tier, _ptr(k), _ptr(v), src_len, _ptr(src_pos), n_tokens, pos_base, _ptr(src_scores),
        ctypes.byref(c), _stream(stream)))


def mikv_decode_attention(q, cache, out, lse, hi_logits=None, ws=None, stream=None):
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    w, nb = _ws(lib.mikv_decode_workspace_bytes(ctypes.byref(c)), q.device, ws)
    _check("mikv_decode_attention", lib.mikv_decode_attention(
        _ptr(q), ctypes.byref(c), _ptr(out), _ptr(lse), _ptr(hi_logits), _ptr(w), nb,
        _stream(stream)))


def mikv_decode_step(q, k_new, v_new, pos, budget_pct, window, policy, cache, out, lse, ws=None,
                     stream=None):
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    w, nb = _ws(lib.mikv_decode_step_workspace_bytes(ctypes.byref(c)), q.device, ws)
    _check("mikv_decode_step", lib.mikv_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), pos, budget_pct, window, policy, ctypes.byref(c),
        _ptr(out), _ptr(lse), _ptr(w), nb, _stream(stream)))


def mikv_output_perturbation(o, o_hat=None, w_o_t=None, y=None, pert=None, ws=None, stream=None):
    """o, o_hat fp32 [B][Hq][D]; w_o_t fp16 [hidden][Hq*D] (W_O transposed, nn.Linear layout);
    y fp32 [B][hidden] and / or pert fp32 [B][Hq] are written."""
    lib = load()
    B, Hq, D = o.shape
    hidden = 0 if w_o_t is None else w_o_t.shape[0]
    w, nb = (None, 0) if w_o_t is None else _ws(lib.mikv_output_perturbation_workspace_bytes(B, Hq, hidden),
                                                o.device, ws)
    _check("mikv_output_perturbation", lib.mikv_output_perturbation(
        _ptr(o), _ptr(o_hat), _ptr(w_o_t), B, Hq, D, hidden, _ptr(y), _ptr(pert), _ptr(w), nb,
        _stream(stream)))


def mikv_topk_attention(q, cache, budget_pct, out, lse=None, keep_idx=None, ws=None, stream=None):
    """Post-attention top-k over a full FP16 cache (all tokens in the important tier)."""
    lib = load()
    c = cache.struct if hasattr(cache, "struct") else cache
    w, nb = _ws(lib.mikv_topk_attention_workspace_bytes(ctypes.byref(c), budget_pct), q.device, ws)
    _check("mikv_topk_attention", lib.mikv_topk_attention(
        _ptr(q), ctypes.byref(c), budget_pct, _ptr(out), _ptr(lse), _ptr(keep_idx), _ptr(w), nb,
        _stream(stream)))


def mikv_channel_quantize(k, bits, codes, meta, stream=None):
    """k fp16 [units, n, D]; codes uint8 [units, n, D*bits/8]; meta fp16 [units, n//64, D, 2]."""
    units, n, D = k.shape
    _check("mikv_channel_quantize", load().mikv_channel_quantize(
        _ptr(k), units, n, D, bits, _ptr(codes), _ptr(meta), _stream(stream)))


def mikv_set_attention_events(begin=None, end=None):
    """Record two torch.cuda.Event objects around the split-K attention launch of every
    following decode call of this thread (None, None clears).  Each event must have been
    recorded once through torch, so that its CUDA event exists."""
    lib = load()
    h = lambda e: None if e is None else e.cuda_event
    _check("mikv_set_attention_events", lib.mikv_set_attention_events(h(begin), h(end)))


WAIT_BITS = {1: "K3 pass 1 (row log-sum-exp)", 2: "K3 pass 2 (column sums)", 4: "K6 (V.W_O norms)",
             8: "K9 (output perturbation)", 16: "mikv_wait_probe"}


def mikv_wait_status(clear=True) -> int:
    """OR of the wait-status bits the tensor-core kernels set since the last clear (0 when no
    bounded mbarrier wait gave up).  Synchronous: call after the work has completed."""
    v = ctypes.c_uint(0)
    _check("mikv_wait_status", load().mikv_wait_status(ctypes.byref(v), int(bool(clear))))
    return v.value


def mikv_wait_probe(polls, arrive, stream=None):
    """One bounded mbarrier wait that gives up (sets wait-status bit 16) unless `arrive`."""
    _check("mikv_wait_probe", load().mikv_wait_probe(int(polls), int(bool(arrive)), _stream(stream)))
