"""Python binding of the OEA MoE decode-layer library (libaware_moe.so).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch supplies device memory (tensors) and streams; the
functions below take torch tensors, check dtypes/devices, and pass raw
pointers to the C ABI declared in include/moe.h under the same names.

There is no fallback: if the shared library is missing or fails to load,
importing the functions raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libaware_moe.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_WORKSPACE, MOE_ERR_UNSUPPORTED = range(6)
MODE_TOPK, MODE_OEA = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
FLAG_NONFINITE_SCORE, FLAG_WAIT_TIMEOUT, FLAG_BAD_INDEX = 0x1, 0x2, 0x4
MAX_TOKENS, MAX_EXPERTS, MAX_SLOTS = 256, 1024, 32

EXPORTED = ["moe_num_slots", "moe_layer_launches", "moe_workspace_bytes", "moe_route", "moe_expert_ffn",
            "moe_expert_ffn_mixed", "moe_pack_int4", "moe_decode_layer", "moe_decode_layer_mixed", "moe_decode_layer_static",
            "moe_device_status", "moe_device_status_static", "moe_set_wait_timeout_us",
            "moe_residency_create", "moe_residency_observe", "moe_residency_flush", "moe_residency_query",
            "moe_residency_destroy", "moe_residency_select", "moe_synth_normal", "moe_status_string", "moe_last_error"]
STATIC_SCRATCH_BYTES = 32 << 20


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status}: {detail}")
        self.status = status


class _Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("B_valid", ctypes.c_int32), ("d", ctypes.c_int32),
                ("N", ctypes.c_int32), ("k", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("k0", ctypes.c_int32), ("p", ctypes.c_float), ("maxP", ctypes.c_int32),
                ("kmax", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class _Mixed(ctypes.Structure):
    _fields_ = [("slot", ctypes.c_void_p), ("q_gate", ctypes.c_void_p), ("q_up", ctypes.c_void_p),
                ("q_down", ctypes.c_void_p), ("n_hot", ctypes.c_int32), ("n_cold", ctypes.c_int32)]


class _ResidencyConfig(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("n_hot", ctypes.c_int32), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("alpha", ctypes.c_double), ("margin", ctypes.c_double), ("update_every", ctypes.c_int32),
                ("max_inflight", ctypes.c_int32)] + \
               [(n, ctypes.c_void_p) for n in ("slot", "counts_acc", "snapshot", "hot_gate", "hot_up", "hot_down",
                                              "host_gate", "host_up", "host_down")]


class _Routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("expert_idx", "weights", "T", "active", "counts", "offsets", "perm",
                 "n_base", "logits")]


_lib = None


def load(path: str | None = None):
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with aware_expert_routing_gb300.build.build()")
    lib = ctypes.CDLL(p)
    V, P = ctypes.c_void_p, ctypes.POINTER
    lib.moe_num_slots.argtypes = [P(_Params)]
    lib.moe_num_slots.restype = ctypes.c_int32
    lib.moe_layer_launches.argtypes = [P(_Params), ctypes.c_int32]
    lib.moe_layer_launches.restype = ctypes.c_int32
    lib.moe_workspace_bytes.argtypes = [P(_Params), ctypes.c_int32]
    lib.moe_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_route.argtypes = [V, V, V, P(_Params), P(_Routing), V, ctypes.c_size_t, V]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_expert_ffn.argtypes = [V, V, V, V, ctypes.c_int32, P(_Params), P(_Routing), V, V,
                                   ctypes.c_size_t, V]
    lib.moe_expert_ffn.restype = ctypes.c_int
    lib.moe_expert_ffn_mixed.argtypes = [V, V, V, V, P(_Mixed), ctypes.c_int32, P(_Params), P(_Routing),
                                         V, V, ctypes.c_size_t, V]
    lib.moe_expert_ffn_mixed.restype = ctypes.c_int
    lib.moe_decode_layer.argtypes = [V, V, V, V, V, V, ctypes.c_int32, P(_Params), P(_Routing), V,
                                     V, ctypes.c_size_t, V]
    lib.moe_decode_layer.restype = ctypes.c_int
    lib.moe_decode_layer_mixed.argtypes = [V, V, V, V, V, V, P(_Mixed), ctypes.c_int32, P(_Params), P(_Routing),
                                           V, V, ctypes.c_size_t, V]
    lib.moe_decode_layer_mixed.restype = ctypes.c_int
    lib.moe_decode_layer_static.argtypes = [V, V, V, V, V, V, ctypes.c_int32, P(_Params), P(_Routing),
                                            V, V]
    lib.moe_decode_layer_static.restype = ctypes.c_int
    lib.moe_device_status.argtypes = [V, V, P(ctypes.c_uint32)]
    lib.moe_device_status.restype = ctypes.c_int
    lib.moe_device_status_static.argtypes = [V, P(ctypes.c_uint32)]
    lib.moe_device_status_static.restype = ctypes.c_int
    lib.moe_pack_int4.argtypes = [V, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, V, V]
    lib.moe_pack_int4.restype = ctypes.c_int
    lib.moe_residency_create.argtypes = [P(_ResidencyConfig), V, P(V), V]
    lib.moe_residency_create.restype = ctypes.c_int
    lib.moe_residency_observe.argtypes = [V, V, V]
    lib.moe_residency_observe.restype = ctypes.c_int
    lib.moe_residency_flush.argtypes = [V, V]
    lib.moe_residency_flush.restype = ctypes.c_int
    lib.moe_residency_query.argtypes = [V, V, V, V]
    lib.moe_residency_query.restype = ctypes.c_int
    lib.moe_residency_destroy.argtypes = [V]
    lib.moe_residency_destroy.restype = ctypes.c_int
    lib.moe_residency_select.argtypes = [V, ctypes.c_int32, ctypes.c_double, V, V, V]
    lib.moe_residency_select.restype = ctypes.c_int32
    lib.moe_set_wait_timeout_us.argtypes = [ctypes.c_uint32]
    lib.moe_set_wait_timeout_us.restype = ctypes.c_int
    lib.moe_synth_normal.argtypes = [V, ctypes.c_int32, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_float, V]
    lib.moe_synth_normal.restype = ctypes.c_int
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_last_error.argtypes = []
    lib.moe_last_error.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


@dataclasses.dataclass
class RouteParams:
    """Mirror of moe_route_params (include/moe.h)."""
    B: int
    d: int
    N: int
    k: int
    mode: int = MODE_TOPK
    k0: int = 0
    p: float = 1.0
    maxP: int = 0
    kmax: int = 0
    B_valid: int = -1
    dtype: int = DTYPE_BF16

    def c(self) -> _Params:
        return _Params(self.B, self.B_valid, self.d, self.N, self.k, self.mode,
                       self.k0 if self.mode == MODE_OEA else self.k, self.p, self.maxP,
                       self.kmax, self.dtype)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == DTYPE_BF16 else torch.float32


def _check(status: int, where: str):
    if status != MOE_OK:
        lib = load()
        raise MoeError(status, where, lib.moe_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def moe_num_slots(params: RouteParams) -> int:
    n = load().moe_num_slots(ctypes.byref(params.c()))
    if n < 0:
        raise MoeError(MOE_ERR_ARG, "moe_num_slots", load().moe_last_error().decode())
    return n


def moe_layer_launches(params: RouteParams, d_ff: int) -> int:
    n = load().moe_layer_launches(ctypes.byref(params.c()), d_ff)
    if n < 0:
        raise MoeError(MOE_ERR_ARG, "moe_layer_launches", load().moe_last_error().decode())
    return n


def moe_workspace_bytes(params: RouteParams, d_ff: int = 0) -> int:
    n = load().moe_workspace_bytes(ctypes.byref(params.c()), d_ff)
    if n == 0:
        raise MoeError(MOE_ERR_ARG, "moe_workspace_bytes", load().moe_last_error().decode())
    return n


def alloc_workspace(params: RouteParams, d_ff: int, device) -> torch.Tensor:
    """A zero-filled workspace tensor of the required size (torch allocates
    with at least 256-byte alignment)."""
    return torch.zeros(moe_workspace_bytes(params, d_ff), dtype=torch.uint8, device=device)


class Routing:
    """Device buffers of moe_routing, allocated with torch."""

    def __init__(self, params: RouteParams, device, with_logits: bool = False,
                 with_n_base: bool = True):
        B, N = params.B, params.N
        ks = moe_num_slots(params)
        i32 = dict(dtype=torch.int32, device=device)
        self.kslots = ks
        self.expert_idx = torch.empty(B, ks, **i32)
        self.weights = torch.empty(B, ks, dtype=torch.float32, device=device)
        self.T = torch.empty(1, **i32)
        self.active = torch.empty(N, **i32)
        self.counts = torch.empty(N, **i32)
        self.offsets = torch.empty(N + 1, **i32)
        self.perm = torch.empty(max(B * ks, 1), **i32)
        self.n_base = torch.empty(max(B, 1), **i32) if with_n_base else None
        self.logits = torch.empty(B, N, dtype=torch.float32, device=device) if with_logits else None

    def c(self) -> _Routing:
        return _Routing(*[_ptr(getattr(self, n)) for n in
                          ("expert_idx", "weights", "T", "active", "counts", "offsets", "perm",
                           "n_base", "logits")])


def _need(t, dtype, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


def moe_route(hidden, w_router, router_bias, params: RouteParams, routing: Routing,
              workspace: torch.Tensor, stream=None):
    dt = params.torch_dtype
    _need(hidden, dt, "hidden")
    _need(w_router, dt, "w_router")
    if router_bias is not None:
        _need(router_bias, torch.float32, "router_bias")
    st = load().moe_route(_ptr(hidden), _ptr(w_router), _ptr(router_bias), ctypes.byref(params.c()),
                          ctypes.byref(routing.c()), _ptr(workspace), workspace.numel(),
                          _stream(stream))
    _check(st, "moe_route")
    return routing


def moe_expert_ffn(hidden, w_gate, w_up, w_down, d_ff: int, params: RouteParams, routing: Routing,
                   out, workspace: torch.Tensor, stream=None):
    dt = params.torch_dtype
    for t, n in ((hidden, "hidden"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down"),
                 (out, "out")):
        _need(t, dt, n)
    st = load().moe_expert_ffn(_ptr(hidden), _ptr(w_gate), _ptr(w_up), _ptr(w_down), d_ff,
                               ctypes.byref(params.c()), ctypes.byref(routing.c()), _ptr(out),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_expert_ffn")
    return out


class MixedExperts:
    """Device buffers of moe_mixed_experts: bf16 hot experts plus INT4 cold
    experts in the packed format of include/moe.h."""

    def __init__(self, slot: torch.Tensor, q_gate, q_up, q_down, n_hot: int, n_cold: int):
        self.slot, self.q_gate, self.q_up, self.q_down = slot, q_gate, q_up, q_down
        self.n_hot, self.n_cold = n_hot, n_cold

    def c(self) -> _Mixed:
        return _Mixed(_ptr(self.slot), _ptr(self.q_gate), _ptr(self.q_up), _ptr(self.q_down),
                      self.n_hot, self.n_cold)


def moe_expert_ffn_mixed(hidden, w_gate, w_up, w_down, mixed: MixedExperts, d_ff: int,
                         params: RouteParams, routing: Routing, out, workspace: torch.Tensor, stream=None):
    for t, n in ((hidden, "hidden"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down"), (out, "out")):
        _need(t, torch.bfloat16, n)
    _need(mixed.slot, torch.int32, "slot")
    st = load().moe_expert_ffn_mixed(_ptr(hidden), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                     ctypes.byref(mixed.c()), d_ff, ctypes.byref(params.c()),
                                     ctypes.byref(routing.c()), _ptr(out), _ptr(workspace),
                                     workspace.numel(), _stream(stream))
    _check(st, "moe_expert_ffn_mixed")
    return out


def int4_image_bytes(rows: int, cols: int) -> int:
    """Bytes of the packed INT4 image of a [rows][cols] matrix."""
    return rows * cols // 2 + rows * (cols // 128) * 2


def moe_pack_int4(w: torch.Tensor, rb: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Packed INT4 image (uint8) of the bf16 matrix w [rows][cols]."""
    _need(w, torch.bfloat16, "w")
    if w.dim() != 2:
        raise ValueError("w must be a matrix")
    rows, cols = w.shape
    n = int4_image_bytes(rows, cols)
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=w.device)
    if not out.is_cuda or out.dtype != torch.uint8 or not out.is_contiguous() or out.numel() < n:
        raise ValueError(f"out must be a contiguous CUDA uint8 tensor of at least {n} bytes")
    _check(load().moe_pack_int4(_ptr(w), rows, cols, rb, _ptr(out), _stream(stream)), "moe_pack_int4")
    return out


MOE_RESIDENT_LO, MOE_RESIDENT_HI, MOE_PROMOTING = 0, 1, 2


def moe_residency_select(S, in_hot, margin: float):
    """The library's selection step on the host: returns (in_hot after the
    swaps, promoted, demoted)."""
    import numpy as np
    S = np.ascontiguousarray(S, dtype=np.float64)
    h = np.ascontiguousarray(in_hot, dtype=np.uint8).copy()
    pro = np.empty(S.size, np.int32)
    dem = np.empty(S.size, np.int32)
    n = load().moe_residency_select(S.ctypes.data, S.size, margin, h.ctypes.data, pro.ctypes.data, dem.ctypes.data)
    if n < 0:
        raise MoeError(MOE_ERR_ARG, "moe_residency_select", "bad arguments")
    return h.astype(bool), [int(x) for x in pro[:n]], [int(x) for x in dem[:n]]


class Residency:
    """moe_residency: which experts keep their bf16 version, changed while
    the layer runs (see include/moe.h).  The caller's buffers: the bf16 pool
    (hot_gate/hot_up/hot_down, n_hot slots, filled with the initial experts
    in order), INT4 images of all N experts, and pinned host bf16 weights of
    all experts (the promotion sources).  The handle table, the count
    accumulator and the pinned snapshot are allocated here with torch."""

    def __init__(self, N: int, d: int, d_ff: int, initial_hot, hot: dict, q: dict, host: dict, alpha: float = 0.9,
                 margin: float = 0.0, update_every: int = 1, max_inflight: int = 4, stream=None):
        import numpy as np
        dev = hot["w_gate"].device
        for t in list(hot.values()):
            _need(t, torch.bfloat16, "bf16 pool")
        for t in host.values():
            if t.is_cuda or not t.is_pinned() or t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError("host weights must be contiguous pinned bf16 CPU tensors")
        self.N, self.n_hot = N, len(initial_hot)
        self.slot = torch.empty(N, dtype=torch.int32, device=dev)
        self.acc = torch.zeros(N, dtype=torch.int32, device=dev)
        self.snapshot = torch.zeros(N, dtype=torch.int32).pin_memory()
        self.hot, self.q, self.host = hot, q, host
        self._cfg = _ResidencyConfig(N, self.n_hot, d, d_ff, alpha, margin, update_every, max_inflight,
                                     self.slot.data_ptr(), self.acc.data_ptr(), self.snapshot.data_ptr(),
                                     hot["w_gate"].data_ptr(), hot["w_up"].data_ptr(), hot["w_down"].data_ptr(),
                                     host["w_gate"].data_ptr(), host["w_up"].data_ptr(), host["w_down"].data_ptr())
        init = np.ascontiguousarray(initial_hot, dtype=np.int32)
        self._init = init
        h = ctypes.c_void_p()
        _check(load().moe_residency_create(ctypes.byref(self._cfg), init.ctypes.data, ctypes.byref(h),
                                           _stream(stream)), "moe_residency_create")
        self._h = h

    def mixed(self) -> "MixedExperts":
        """The expert descriptor for the mixed layer calls."""
        return MixedExperts(self.slot, self.q["w_gate"], self.q["w_up"], self.q["w_down"], self.n_hot, self.N)

    def observe(self, counts: torch.Tensor, stream=None):
        _need(counts, torch.int32, "counts")
        _check(load().moe_residency_observe(self._h, _ptr(counts), _stream(stream)), "moe_residency_observe")

    def flush(self, stream=None):
        _check(load().moe_residency_flush(self._h, _stream(stream)), "moe_residency_flush")

    def query(self):
        """(state [N], scores [N], stats dict)."""
        import numpy as np
        st = np.empty(self.N, np.int32)
        sc = np.empty(self.N, np.float64)
        stats = np.empty(5, np.uint64)
        _check(load().moe_residency_query(self._h, st.ctypes.data, sc.ctypes.data, stats.ctypes.data),
               "moe_residency_query")
        keys = ("calls", "updates", "promotions", "demotions", "pending")
        return st, sc, {k: int(v) for k, v in zip(keys, stats)}

    def close(self):
        if getattr(self, "_h", None):
            load().moe_residency_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ema_hot_set(counts, n_hot: int, alpha: float = 0.9) -> "np.ndarray":
    """Hot experts of a routing trace (DynaExq page, section 2.5): per step
    S <- alpha * S + (1 - alpha) * c, S starting at 0, then the n_hot experts
    with the largest S (ties to the lower id).  `counts` is [steps][N]
    (selections per expert per step).  Host-side policy arithmetic."""
    import numpy as np
    c = np.asarray(counts, dtype=np.float64)
    S = np.zeros(c.shape[1])
    for row in c:
        S = alpha * S + (1.0 - alpha) * row
    order = sorted(range(c.shape[1]), key=lambda e: (-S[e], e))
    return np.array(sorted(order[:n_hot]), dtype=np.int64)


def moe_decode_layer(hidden, w_router, router_bias, w_gate, w_up, w_down, d_ff: int,
                     params: RouteParams, routing: Routing, out, workspace: torch.Tensor,
                     stream=None):
    dt = params.torch_dtype
    for t, n in ((hidden, "hidden"), (w_router, "w_router"), (w_gate, "w_gate"), (w_up, "w_up"),
                 (w_down, "w_down"), (out, "out")):
        _need(t, dt, n)
    if router_bias is not None:
        _need(router_bias, torch.float32, "router_bias")
    st = load().moe_decode_layer(_ptr(hidden), _ptr(w_router), _ptr(router_bias), _ptr(w_gate),
                                 _ptr(w_up), _ptr(w_down), d_ff, ctypes.byref(params.c()),
                                 ctypes.byref(routing.c()), _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(st, "moe_decode_layer")
    return out


def moe_decode_layer_mixed(hidden, w_router, router_bias, w_gate, w_up, w_down, mixed: MixedExperts,
                           d_ff: int, params: RouteParams, routing: Routing, out, workspace: torch.Tensor,
                           stream=None):
    """The whole layer with bf16 hot and INT4 cold experts in one call."""
    for t, n in ((hidden, "hidden"), (w_router, "w_router"), (w_gate, "w_gate"), (w_up, "w_up"),
                 (w_down, "w_down"), (out, "out")):
        _need(t, torch.bfloat16, n)
    if router_bias is not None:
        _need(router_bias, torch.float32, "router_bias")
    _need(mixed.slot, torch.int32, "slot")
    st = load().moe_decode_layer_mixed(_ptr(hidden), _ptr(w_router), _ptr(router_bias), _ptr(w_gate),
                                       _ptr(w_up), _ptr(w_down), ctypes.byref(mixed.c()), d_ff,
                                       ctypes.byref(params.c()), ctypes.byref(routing.c()), _ptr(out),
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_decode_layer_mixed")
    return out


def moe_decode_layer_static(hidden, w_router, router_bias, w_gate, w_up, w_down, d_ff: int,
                            params: RouteParams, routing: Routing, out, stream=None):
    """moe_decode_layer without a workspace, for callers that cannot
    allocate device memory: the scratch is the library's fixed device array
    of STATIC_SCRATCH_BYTES (see include/moe.h for its limits)."""
    dt = params.torch_dtype
    for t, n in ((hidden, "hidden"), (w_router, "w_router"), (w_gate, "w_gate"), (w_up, "w_up"),
                 (w_down, "w_down"), (out, "out")):
        _need(t, dt, n)
    if router_bias is not None:
        _need(router_bias, torch.float32, "router_bias")
    st = load().moe_decode_layer_static(_ptr(hidden), _ptr(w_router), _ptr(router_bias), _ptr(w_gate),
                                        _ptr(w_up), _ptr(w_down), d_ff, ctypes.byref(params.c()),
                                        ctypes.byref(routing.c()), _ptr(out), _stream(stream))
    _check(st, "moe_decode_layer_static")
    return out


def moe_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream; returns and clears the device flag word."""
    f = ctypes.c_uint32(0)
    load().moe_device_status(_ptr(workspace), _stream(stream), ctypes.byref(f))
    return int(f.value)


def moe_device_status_static(stream=None) -> int:
    """Synchronises the stream; returns and clears the flag word of the
    calls of moe_decode_layer_static on the current device."""
    f = ctypes.c_uint32(0)
    load().moe_device_status_static(_stream(stream), ctypes.byref(f))
    return int(f.value)


def moe_set_wait_timeout_us(microseconds: int):
    """Bound of every in-kernel wait (0: the default of two seconds)."""
    _check(load().moe_set_wait_timeout_us(int(microseconds)), "moe_set_wait_timeout_us")


def moe_synth_normal(dst: torch.Tensor, seed: int, scale: float, start: int = 0, stream=None):
    """Fill `dst` (bf16 or fp32) with the seeded synthetic stream."""
    if dst.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif dst.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise ValueError("dst must be bf16 or fp32")
    if not dst.is_cuda or not dst.is_contiguous():
        raise ValueError("dst must be a contiguous CUDA tensor")
    st = load().moe_synth_normal(_ptr(dst), dt, dst.numel(), start, seed & ((1 << 64) - 1),
                                 ctypes.c_float(scale), _stream(stream))
    _check(st, "moe_synth_normal")
    return dst
