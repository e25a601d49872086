"""Python binding of the GB300 MoE decode library (libmoedecode.so).

Argument marshalling only: every computation runs in the library's CUDA
kernels. PyTorch provides device memory and streams. The names follow the C
ABI in ``include/moe_decode.h``. If the library has not been built, importing
works but every call raises ``RuntimeError``; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoedecode.so")

DEC_OK, DEC_ERR_INVALID_ARG, DEC_ERR_UNSUPPORTED, DEC_ERR_CUDA, DEC_ERR_TIMEOUT = range(5)
VARIANT_AUTO, VARIANT_SMALL_M, VARIANT_SPLIT_K = 0, 1, 2

_lib = None


class DecodeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _load().dec_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


def build() -> str:
    """Compile the CUDA library in-tree for sm_103a (nvcc)."""
    from . import _build
    return _build.build()


class _LayerWeights(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("N_in", ctypes.c_int), ("K_out", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("I", ctypes.c_int), ("eps", ctypes.c_float)] + \
               [(n, ctypes.c_void_p) for n in ("gamma1", "W_in", "W_o", "gamma2", "W_r", "Wg", "Wu", "Wd",
                                               "Wg_s", "Wu_s", "Wd_s", "prefetch_next")] + \
               [("prefetch_bytes", ctypes.c_size_t)]


class _MoeWeights(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
                ("eps", ctypes.c_float)] + \
               [(n, ctypes.c_void_p) for n in ("gamma", "W_r", "Wg", "Wu", "Wd", "Wg_s", "Wu_s", "Wd_s")]


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class _LayerTrace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("h1", "idx", "w", "scores")]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_layers_gb300.build() "
                           "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_float
    sig = {
        "dec_create": [ctypes.POINTER(P), I],
        "dec_destroy": [P],
        "dec_workspace_init": [P, P, Z, P],
        "dec_set_wait_limit_ns": [P, U64],
        "dec_set_pdl": [P, I],
        "dec_set_force_variant": [P, I],
        "dec_set_shared_sms": [P, I],
        "dec_set_l2_ahead": [P, I],
        "dec_test_set_moe_front": [P, I],
        "dec_test_set_engine_finish": [P, I],
        "dec_check_device_error": [P],
        "dec_linear_workspace_size": [P, I, I, I, ctypes.POINTER(Z)],
        "dec_linear": [P, P, I, P, P, I, I, I, P, Z, P],
        "dec_linear_residual": [P, P, I, P, P, P, I, I, I, P, Z, P],
        "dec_linear_noalloc": [P, P, I, P, P, P, I, I, I, P],
        "dec_rmsnorm": [P, P, P, P, I, I, F, P],
        "moe_route_topk_workspace_size": [P, I, I, I, ctypes.POINTER(Z)],
        "moe_route_topk": [P, P, P, I, I, I, I, P, P, P, P, Z, P],
        "moe_experts_workspace_size": [P, I, I, I, I, I, ctypes.POINTER(Z)],
        "moe_experts": [P, P, P, P, I, I, P, P, P, I, I, I, P, P, P, P, P, P, Z, P],
        "moe_layer_workspace_size": [P, ctypes.POINTER(_MoeWeights), I, ctypes.POINTER(Z)],
        "moe_layer": [P, ctypes.POINTER(_MoeWeights), P, P, P, I, P, P, P, P, Z, P],
        "decode_layer_workspace_size": [P, ctypes.POINTER(_LayerWeights), I, ctypes.POINTER(Z)],
        "decode_layer": [P, ctypes.POINTER(_LayerWeights), P, I, ctypes.POINTER(_LayerTrace), P, Z, P],
        "dec_prefetch_l2": [P, P, Z, P],
        "dec_test_wait_timeout": [P, P],
        "dec_test_routing_wait_timeout": [P, I, P],
        "dec_test_delayed_copy": [P, P, P, Z, U64, P],
        "dec_test_occupy_sms": [P, I, U64, P],
        "dec_set_profiling": [P, I],
        "dec_profile_read": [P, ctypes.POINTER(_KernelTime), I, ctypes.POINTER(I)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.dec_status_string.argtypes = [ctypes.c_int]
    lib.dec_status_string.restype = ctypes.c_char_p
    lib.dec_last_variant.argtypes = [P]
    lib.dec_last_variant.restype = ctypes.c_int
    lib.dec_last_expert_variant.argtypes = [P]
    lib.dec_last_expert_variant.restype = ctypes.c_int
    lib.dec_launch_count.argtypes = [P]
    lib.dec_launch_count.restype = ctypes.c_uint64
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != DEC_OK:
        raise DecodeError(status, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _require(t, dtype, name: str, ndim: Optional[int] = None):
    import torch
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t


def _rows(t, name: str) -> int:
    """Row stride (elements) of a 2-D tensor whose rows are contiguous."""
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: rows must be contiguous")
    return t.stride(0) if t.dim() == 2 else t.shape[-1]


class Handle:
    """Owns a dec_handle (side streams, events, device error word) and cached workspaces."""

    def __init__(self, device: int = 0):
        lib = _load()
        h = ctypes.c_void_p()
        _check(lib.dec_create(ctypes.byref(h), int(device)), "dec_create")
        self._h = h
        self.device = int(device)
        self._ws = {}

    @property
    def ptr(self):
        return self._h

    def close(self) -> None:
        if self._h:
            _load().dec_destroy(self._h)
            self._h = ctypes.c_void_p()
            self._ws.clear()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, key, nbytes: int, layout=None):
        """A workspace of at least nbytes, reused per key. It is zeroed when it
        is created and whenever the layout (entry point and shape) that uses it
        changes, as the C ABI requires; calls with the same layout leave it ready."""
        import torch
        t, last = self._ws.get(key, (None, None))
        if t is None or t.numel() < nbytes:
            t = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=f"cuda:{self.device}")
        elif layout != last:
            t.zero_()
        self._ws[key] = (t, layout)
        return t

    def set_force_variant(self, v: int) -> None:
        _check(_load().dec_set_force_variant(self._h, int(v)), "dec_set_force_variant")

    def set_shared_sms(self, n: int) -> None:
        """0: automatic SM share by expected bytes; -1: every SM, overlapped; n > 0: a fixed n-SM partition."""
        _check(_load().dec_set_shared_sms(self._h, int(n)), "dec_set_shared_sms")

    def test_set_moe_front(self, enable: bool) -> None:
        """Test hook: False runs the path taken where an MoE front does not apply."""
        _check(_load().dec_test_set_moe_front(self._h, 1 if enable else 0), "dec_test_set_moe_front")

    def test_set_engine_finish(self, mode: int) -> None:
        """Test hook: how the split-K kernel finishes split tiles (0 default; 1, 2 the fallback paths)."""
        _check(_load().dec_test_set_engine_finish(self._h, int(mode)), "dec_test_set_engine_finish")

    def set_l2_ahead(self, nbytes: int) -> None:
        _check(_load().dec_set_l2_ahead(self._h, int(nbytes)), "dec_set_l2_ahead")

    def set_pdl(self, enable: bool) -> None:
        _check(_load().dec_set_pdl(self._h, 1 if enable else 0), "dec_set_pdl")

    def set_wait_limit_ns(self, ns: int) -> None:
        _check(_load().dec_set_wait_limit_ns(self._h, int(ns)), "dec_set_wait_limit_ns")

    @property
    def last_variant(self) -> int:
        return _load().dec_last_variant(self._h)

    @property
    def last_expert_variant(self) -> int:
        return _load().dec_last_expert_variant(self._h)

    def check_device_error(self) -> int:
        return _load().dec_check_device_error(self._h)

    def set_profiling(self, enable: bool) -> None:
        _check(_load().dec_set_profiling(self._h, 1 if enable else 0), "dec_set_profiling")

    def profile_read(self) -> dict:
        """{kernel tag: (launches, total_ms)} since the last read (synchronises)."""
        buf = (_KernelTime * 64)()
        n = ctypes.c_int()
        _check(_load().dec_profile_read(self._h, buf, 64, ctypes.byref(n)), "dec_profile_read")
        return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}

    @property
    def launch_count(self) -> int:
        return int(_load().dec_launch_count(self._h))


# ---------------------------------------------------------------------------- projections
def dec_linear(h: Handle, x, W, y=None, stream=None, ws=None):
    """y = x W^T (bf16). x [M,K] (rows may be strided), W [N,K]."""
    import torch
    lib = _load()
    _require(x, torch.bfloat16, "x", 2)
    _require(W, torch.bfloat16, "W", 2)
    M, K = x.shape
    N = W.shape[0]
    if not W.is_contiguous():
        raise ValueError("W must be contiguous")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    nb = ctypes.c_size_t()
    _check(lib.dec_linear_workspace_size(h.ptr, M, N, K, ctypes.byref(nb)), "dec_linear_workspace_size")
    ws = h.workspace(("linear", id(stream)), nb.value, ("linear", M, N, K)) if ws is None else ws
    _check(lib.dec_linear(h.ptr, _ptr(x), _rows(x, "x"), _ptr(W), _ptr(y), M, N, K, _ptr(ws), ws.numel(),
                          _stream(stream)), "dec_linear")
    return y


def dec_linear_residual(h: Handle, x, W, r, out=None, stream=None, ws=None):
    """out = r + x W^T (bf16); out may be r itself."""
    import torch
    lib = _load()
    _require(x, torch.bfloat16, "x", 2)
    _require(W, torch.bfloat16, "W", 2)
    _require(r, torch.bfloat16, "r", 2)
    M, K = x.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    nb = ctypes.c_size_t()
    _check(lib.dec_linear_workspace_size(h.ptr, M, N, K, ctypes.byref(nb)), "dec_linear_workspace_size")
    ws = h.workspace(("linear", id(stream)), nb.value, ("linear", M, N, K)) if ws is None else ws
    _check(lib.dec_linear_residual(h.ptr, _ptr(x), _rows(x, "x"), _ptr(W), _ptr(r), _ptr(out), M, N, K, _ptr(ws),
                                   ws.numel(), _stream(stream)), "dec_linear_residual")
    return out


def dec_linear_noalloc(h: Handle, x, W, r=None, out=None, stream=None):
    """out = [r +] x W^T through the entry point that takes no workspace and
    allocates nothing (its scratch is a static device array in the library)."""
    import torch
    _require(x, torch.bfloat16, "x", 2)
    _require(W, torch.bfloat16, "W", 2)
    M, K = x.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(_load().dec_linear_noalloc(h.ptr, _ptr(x), _rows(x, "x"), _ptr(W), _ptr(r), _ptr(out), M, N, K,
                                      _stream(stream)), "dec_linear_noalloc")
    return out


def dec_rmsnorm(h: Handle, x, gamma, y=None, eps: float = 1e-6, stream=None):
    import torch
    _require(x, torch.bfloat16, "x", 2)
    _require(gamma, torch.bfloat16, "gamma", 1)
    M, H = x.shape
    if y is None:
        y = torch.empty_like(x)
    _check(_load().dec_rmsnorm(h.ptr, _ptr(x), _ptr(gamma), _ptr(y), M, H, ctypes.c_float(eps), _stream(stream)),
           "dec_rmsnorm")
    return y


# ---------------------------------------------------------------------------- router / experts
def moe_route_topk(h: Handle, x, Wr, k: int, want_scores: bool = True, stream=None):
    """Returns (idx int32 [M,k], w fp32 [M,k], scores fp32 [M,E] or None)."""
    import torch
    lib = _load()
    _require(x, torch.bfloat16, "x", 2)
    _require(Wr, torch.float32, "Wr", 2)
    M, H = x.shape
    E = Wr.shape[0]
    idx = torch.empty((M, k), dtype=torch.int32, device=x.device)
    w = torch.empty((M, k), dtype=torch.float32, device=x.device)
    scores = torch.empty((M, E), dtype=torch.float32, device=x.device) if want_scores else None
    nb = ctypes.c_size_t()
    _check(lib.moe_route_topk_workspace_size(h.ptr, M, H, E, ctypes.byref(nb)), "moe_route_topk_workspace_size")
    ws = h.workspace(("router", id(stream)), nb.value, ("router", M, H, E))
    _check(lib.moe_route_topk(h.ptr, _ptr(x), _ptr(Wr), M, H, E, int(k), _ptr(idx), _ptr(w), _ptr(scores),
                              _ptr(ws), ws.numel(), _stream(stream)), "moe_route_topk")
    return idx, w, scores


def moe_experts(h: Handle, x, idx, w, Wg, Wu, Wd, shared: Optional[Sequence] = None, residual=None, out=None,
                stream=None):
    """out = [residual +] sum_j w_j E_idx_j(x) [+ S(x)] (bf16 [M,H])."""
    import torch
    lib = _load()
    _require(x, torch.bfloat16, "x", 2)
    _require(idx, torch.int32, "idx", 2)
    _require(w, torch.float32, "w", 2)
    for n, t in (("Wg", Wg), ("Wu", Wu), ("Wd", Wd)):
        _require(t, torch.bfloat16, n, 3)
    M, H = x.shape
    k = idx.shape[1]
    E, I, _ = Wg.shape
    sg, su, sd = (None, None, None) if shared is None else shared
    if out is None:
        out = torch.empty_like(x)
    nb = ctypes.c_size_t()
    _check(lib.moe_experts_workspace_size(h.ptr, M, k, E, H, I, ctypes.byref(nb)), "moe_experts_workspace_size")
    ws = h.workspace(("experts", id(stream)), nb.value, ("experts", M, k, E, H, I))
    _check(lib.moe_experts(h.ptr, _ptr(x), _ptr(idx), _ptr(w), M, k, _ptr(Wg), _ptr(Wu), _ptr(Wd), E, H, I,
                           _ptr(sg), _ptr(su), _ptr(sd), _ptr(residual), _ptr(out), _ptr(ws), ws.numel(),
                           _stream(stream)), "moe_experts")
    return out


@dataclass
class MoeWeights:
    """Device tensors of one MoE layer (see dec_moe_weights); gamma None: no RMSNorm."""
    W_r: object
    Wg: object
    Wu: object
    Wd: object
    Wg_s: object = None
    Wu_s: object = None
    Wd_s: object = None
    gamma: object = None
    k: int = 8
    eps: float = 1e-6

    def c_struct(self) -> _MoeWeights:
        E, I, H = self.Wg.shape
        s = _MoeWeights()
        s.H, s.E, s.k, s.I, s.eps = H, E, self.k, I, self.eps
        for n in ("gamma", "W_r", "Wg", "Wu", "Wd", "Wg_s", "Wu_s", "Wd_s"):
            setattr(s, n, _ptr(getattr(self, n)))
        return s


def moe_layer_workspace_size(h: Handle, weights: MoeWeights, M: int) -> int:
    nb = ctypes.c_size_t()
    cw = weights.c_struct()
    _check(_load().moe_layer_workspace_size(h.ptr, ctypes.byref(cw), int(M), ctypes.byref(nb)),
           "moe_layer_workspace_size")
    return nb.value


def moe_layer(h: Handle, weights: MoeWeights, x, residual=None, out=None, trace=False, stream=None, ws=None,
              _cw=None):
    """out = [residual +] MoE([RMSNorm](x)) (bf16 [M,H]): routing and experts in one call.

    trace=True also returns a dict of new device tensors with the routing
    (idx, w, scores); trace may be a dict of preallocated tensors (any of those
    keys). Returns out, or (out, trace dict)."""
    import torch
    lib = _load()
    _require(x, torch.bfloat16, "x", 2)
    M = x.shape[0]
    cw = weights.c_struct() if _cw is None else _cw
    if out is None:
        out = torch.empty_like(x)
    if ws is None:
        ws = h.workspace(("moe_layer", id(stream)), moe_layer_workspace_size(h, weights, M),
                         ("moe_layer", M, cw.H, cw.E, cw.k, cw.I))
    tr = None
    if trace is True:
        tr = dict(idx=torch.empty((M, cw.k), dtype=torch.int32, device=x.device),
                  w=torch.empty((M, cw.k), dtype=torch.float32, device=x.device),
                  scores=torch.empty((M, cw.E), dtype=torch.float32, device=x.device))
    elif isinstance(trace, dict):
        tr = trace
    g = (lambda n: None) if tr is None else tr.get
    _check(lib.moe_layer(h.ptr, ctypes.byref(cw), _ptr(x), _ptr(residual), _ptr(out), M, _ptr(g("idx")),
                         _ptr(g("w")), _ptr(g("scores")), _ptr(ws), ws.numel(), _stream(stream)), "moe_layer")
    return out if tr is None else (out, tr)


@dataclass
class LayerWeights:
    """Device tensors of one decode layer (see dec_layer_weights)."""
    gamma1: object
    W_in: object
    W_o: object
    gamma2: object
    W_r: object
    Wg: object
    Wu: object
    Wd: object
    Wg_s: object = None
    Wu_s: object = None
    Wd_s: object = None
    k: int = 8
    k_out: Optional[int] = None
    eps: float = 1e-6
    prefetch_next: object = None
    prefetch_bytes: int = 0

    def c_struct(self) -> _LayerWeights:
        E, I, H = self.Wg.shape
        s = _LayerWeights()
        s.H, s.N_in = H, self.W_in.shape[0]
        s.K_out = self.W_o.shape[1] if self.k_out is None else self.k_out
        s.E, s.k, s.I, s.eps = E, self.k, I, self.eps
        for n in ("gamma1", "W_in", "W_o", "gamma2", "W_r", "Wg", "Wu", "Wd", "Wg_s", "Wu_s", "Wd_s",
                  "prefetch_next"):
            setattr(s, n, _ptr(getattr(self, n)))
        s.prefetch_bytes = int(self.prefetch_bytes)
        return s


def decode_layer_workspace_size(h: Handle, weights: LayerWeights, M: int) -> int:
    nb = ctypes.c_size_t()
    cw = weights.c_struct()
    _check(_load().decode_layer_workspace_size(h.ptr, ctypes.byref(cw), int(M), ctypes.byref(nb)),
           "decode_layer_workspace_size")
    return nb.value


def decode_layer(h: Handle, weights: LayerWeights, hidden, trace=False, stream=None, ws=None, _cw=None):
    """One decode layer in place on hidden bf16 [M,H].

    trace=True returns a dict of new device tensors with the intermediates
    (h1, idx, w, scores); trace may also be a dict of preallocated tensors
    (any of those keys, others omitted) that receive them."""
    import torch
    lib = _load()
    _require(hidden, torch.bfloat16, "hidden", 2)
    M = hidden.shape[0]
    cw = weights.c_struct() if _cw is None else _cw
    if ws is None:
        ws = h.workspace(("layer", id(stream)), decode_layer_workspace_size(h, weights, M),
                         ("layer", M, cw.H, cw.N_in, cw.K_out, cw.E, cw.k, cw.I))
    tr = None
    out = None
    if trace is True:
        out = dict(h1=torch.empty_like(hidden),
                   idx=torch.empty((M, cw.k), dtype=torch.int32, device=hidden.device),
                   w=torch.empty((M, cw.k), dtype=torch.float32, device=hidden.device),
                   scores=torch.empty((M, cw.E), dtype=torch.float32, device=hidden.device))
    elif isinstance(trace, dict):
        out = trace
    if out is not None:
        tr = _LayerTrace()
        tr.h1, tr.idx, tr.w, tr.scores = (_ptr(out.get(n)) for n in ("h1", "idx", "w", "scores"))
    _check(lib.decode_layer(h.ptr, ctypes.byref(cw), _ptr(hidden), M, ctypes.byref(tr) if tr is not None else None,
                            _ptr(ws), ws.numel(), _stream(stream)), "decode_layer")
    return out


def dec_prefetch_l2(h: Handle, t, nbytes: Optional[int] = None, stream=None) -> None:
    n = t.numel() * t.element_size() if nbytes is None else int(nbytes)
    _check(_load().dec_prefetch_l2(h.ptr, _ptr(t), n, _stream(stream)), "dec_prefetch_l2")


def test_wait_timeout(h: Handle, stream=None) -> None:
    _check(_load().dec_test_wait_timeout(h.ptr, _stream(stream)), "dec_test_wait_timeout")

def test_routing_wait_timeout(h: Handle, tokens: int = 1, stream=None) -> None:
    _check(_load().dec_test_routing_wait_timeout(h.ptr, int(tokens), _stream(stream)),
           "dec_test_routing_wait_timeout")


def test_occupy_sms(h: Handle, ctas: int, hold_ns: int, stream=None) -> None:
    """Hold `ctas` SMs for hold_ns with a sleeping kernel on `stream` (a test hook)."""
    _check(_load().dec_test_occupy_sms(h.ptr, int(ctas), int(hold_ns), _stream(stream)), "dec_test_occupy_sms")


def test_delayed_copy(h: Handle, dst, src, delay_ns: int, stream=None) -> None:
    n = src.numel() * src.element_size()
    _check(_load().dec_test_delayed_copy(h.ptr, _ptr(dst), _ptr(src), n, int(delay_ns), _stream(stream)),
           "dec_test_delayed_copy")
