"""CPU oracle of the OEA MoE decode layer (test infrastructure only).

Thin ctypes wrapper around ``oracle.c``: plain single-threaded loops, fp64
sums, routing decisions in fp32.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg use this package; the library never does, and
nothing here imports the library.

Each function names the passage it follows in its docstring; ``oracle.c``
holds the full list.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TOPK, OEA = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_router_logits.argtypes = [P, P, P, i, i, i, P]
            lib.oracle_router_logits.restype = None
            lib.oracle_route.argtypes = [P, i, i, i, i, i, ctypes.c_float, i, i, i, P,
                                         P, P, P, P, P, P, P, P]
            lib.oracle_route.restype = i
            lib.oracle_policy_k0.argtypes = [i, i, ctypes.POINTER(ctypes.c_float)]
            lib.oracle_policy_k0.restype = i
            lib.oracle_expert_ffn.argtypes = [P, P, P, P, i, i, P]
            lib.oracle_expert_ffn.restype = None
            lib.oracle_moe_experts.argtypes = [P, P, P, P, i, i, i, i, P, P, P]
            lib.oracle_moe_experts.restype = None
            lib.oracle_dequant_int4.argtypes = [P, i, i, i, P]
            lib.oracle_dequant_int4.restype = None
            lib.oracle_ema_update.argtypes = [P, P, i, ctypes.c_double]
            lib.oracle_ema_update.restype = None
            lib.oracle_hot_select.argtypes = [P, i, ctypes.c_double, P, P, P]
            lib.oracle_hot_select.restype = i
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def router_logits(x, w_router, bias=None) -> np.ndarray:
    """fp64 router scores x . W_router^T + bias (OEA page, section 2 Q2)."""
    x, w_router = _f32(x), _f32(w_router)
    B, d = x.shape
    N = w_router.shape[0]
    bias = _f32(bias) if bias is not None else None
    out = np.empty((B, N), np.float64)
    _load().oracle_router_logits(_ptr(x), _ptr(w_router), _ptr(bias), B, N, d, _ptr(out))
    return out


def policy_k0(B_valid: int, k: int, p: float = 1.0) -> tuple:
    """(k0, p) of the batch-size-dependent policy (OEA page, section 7,
    implementation detail 2): plain top-k for at most one real token,
    ceil(5k/8) below 16 tokens, ceil(3k/8) from 16 tokens on."""
    pp = ctypes.c_float(p)
    k0 = _load().oracle_policy_k0(B_valid, k, ctypes.byref(pp))
    return k0, float(pp.value)


def route(logits, mode: int, k: int, k0: int | None = None, p: float = 1.0,
          maxP: int | None = None, kmax: int | None = None,
          B_valid: int | None = None, nbase=None) -> dict:
    """Plain top-k or OEA routing of fp32 logits (OEA page, sections 2-5, 7).

    k0 <= 0 (OEA) takes k0 from ``policy_k0``.  ``nbase`` (OEA, optional,
    [B] ints): phase 1 uses these n_i for the real tokens instead of the
    top-p count.
    Returns idx [B, kslots] int32, w [B, kslots] fp64, nbase [B], T,
    counts [N], offsets [N+1], active [T], perm [sum counts].
    """
    logits = _f32(logits)
    B, N = logits.shape
    k0 = k if k0 is None else k0
    maxP = N if maxP is None else maxP
    kmax = k if kmax is None else kmax
    B_valid = B if B_valid is None else B_valid
    kslots = k if mode == TOPK else kmax
    nb_in = None if nbase is None else np.ascontiguousarray(nbase, dtype=np.int32)
    if nb_in is not None and nb_in.shape != (B,):
        raise ValueError("nbase must hold one n_i per token")
    idx = np.empty((B, kslots), np.int32)
    w = np.empty((B, kslots), np.float64)
    nbase = np.empty(B, np.int32)
    T = np.zeros(1, np.int32)
    counts = np.empty(N, np.int32)
    offsets = np.empty(N + 1, np.int32)
    active = np.empty(N, np.int32)
    perm = np.empty(max(B * kslots, 1), np.int32)
    rc = _load().oracle_route(_ptr(logits), B, N, mode, k, k0, ctypes.c_float(p), maxP,
                              kmax, B_valid, _ptr(nb_in), _ptr(idx), _ptr(w), _ptr(nbase),
                              _ptr(T), _ptr(counts), _ptr(offsets), _ptr(active), _ptr(perm))
    if rc != 0:
        raise ValueError("oracle_route: invalid arguments")
    t = int(T[0])
    return {"idx": idx, "w": w, "nbase": nbase, "T": t, "counts": counts,
            "offsets": offsets, "active": active[:t].copy(),
            "perm": perm[:int(offsets[N])].copy(), "kslots": kslots}


def expert_ffn(x, w_gate, w_up, w_down) -> np.ndarray:
    """One SwiGLU expert on one token, fp64: W_down (silu(W_gate x) * (W_up x))."""
    x, w_gate, w_up, w_down = map(_f32, (x, w_gate, w_up, w_down))
    F, d = w_gate.shape
    y = np.empty(d, np.float64)
    _load().oracle_expert_ffn(_ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), d, F, _ptr(y))
    return y


def moe_experts(x, w_gate, w_up, w_down, idx, w) -> np.ndarray:
    """Expert stage + weighted combine, fp64, slot order (OEA page, section 2 Q2)."""
    x, w_gate, w_up, w_down = map(_f32, (x, w_gate, w_up, w_down))
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    B, d = x.shape
    F = w_gate.shape[1]
    out = np.empty((B, d), np.float64)
    _load().oracle_moe_experts(_ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), B, d, F,
                               idx.shape[1], _ptr(idx), _ptr(w), _ptr(out))
    return out


def dequant_int4(packed, rows: int, cols: int, rb: int) -> np.ndarray:
    """INT4 group-wise codes times bf16 scales -> fp32, from the packed
    cold-expert byte format (DynaExq page, section 3.2, INT4 tier)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty((rows, cols), np.float32)
    _load().oracle_dequant_int4(_ptr(packed), rows, cols, rb, _ptr(out))
    return out


def moe_layer(x, w_router, w_gate, w_up, w_down, bias, mode, k, k0=None, p=1.0,
              maxP=None, kmax=None, B_valid=None) -> dict:
    """Whole layer from the oracle's own logits (fp64 sums, rounded to fp32
    for the routing decisions)."""
    lg = router_logits(x, w_router, bias)
    r = route(lg.astype(np.float32), mode, k, k0, p, maxP, kmax, B_valid)
    r["logits"] = lg
    r["out"] = moe_experts(x, w_gate, w_up, w_down, r["idx"], r["w"])
    return r


def ema_update(S, counts, alpha: float) -> np.ndarray:
    """One hotness update S <- alpha S + (1 - alpha) c (DynaExq page,
    section 2.5); returns the new scores."""
    S = np.array(S, dtype=np.float64)
    c = np.ascontiguousarray(counts, dtype=np.float64)
    _load().oracle_ema_update(_ptr(S), _ptr(c), S.size, alpha)
    return S


def hot_select(S, in_hot, margin: float):
    """The high-precision set after one selection with hysteresis (DynaExq
    page, sections 2.5 and 3.5): returns (new in_hot [N] bool, promoted,
    demoted), the swaps in the order they are made."""
    S = np.ascontiguousarray(S, dtype=np.float64)
    h = np.ascontiguousarray(in_hot, dtype=np.uint8).copy()
    N = S.size
    pro = np.empty(N, np.int32)
    dem = np.empty(N, np.int32)
    n = _load().oracle_hot_select(_ptr(S), N, margin, _ptr(h), _ptr(pro), _ptr(dem))
    return h.astype(bool), [int(x) for x in pro[:n]], [int(x) for x in dem[:n]]
