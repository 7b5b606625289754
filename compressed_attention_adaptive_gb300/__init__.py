"""Python binding of libmita.so, the GB300 MiTA attention forward pass.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libmita.so``; PyTorch supplies device memory and the stream. The
entry points carry the names of the C ABI in ``include/mita.h``:
``mita_workspace_size``, ``mita_landmarks``, ``mita_select``,
``mita_forward``, ``mita_host_buffer_size``, ``mita_forward_host``,
``mita_forward_static``, ``mita_backward_workspace_size``, ``mita_backward``,
``mita_device_status``, ``mita_uses_tensor_cores``.

The library must be built first (``python -c "import __graft_entry__ as g;
g.build()"``); calling an entry point without it raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmita.so")
_lib = None

F32, BF16 = 0, 1
FLAG_NO_SHARED, FLAG_SIMT, FLAG_CAUSAL = 1, 2, 4
TESTFLAG_STALL_PRODUCER = 1 << 31  # fault test only (see include/mita.h)
STATUS = {0: "MITA_OK", 1: "MITA_ERR_INVALID_ARG", 2: "MITA_ERR_UNSUPPORTED", 3: "MITA_ERR_WORKSPACE",
          4: "MITA_ERR_CUDA", 5: "MITA_ERR_TIMEOUT", 6: "MITA_ERR_BOUNDS"}


class MitaError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__("%s: %s" % (STATUS.get(status, status), detail))
        self.status = status
        self.detail = detail


class _CParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
                ("m", ctypes.c_int), ("k", ctypes.c_int), ("s", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int), ("lm_h", ctypes.c_int), ("lm_w", ctypes.c_int),
                ("scale", ctypes.c_float), ("flags", ctypes.c_uint), ("dtype", ctypes.c_int)]


@dataclasses.dataclass
class Params:
    """Mirror of ``mita_params`` (see include/mita.h)."""
    B: int
    H: int
    N: int
    d: int
    m: int
    k: int
    s: int
    grid_h: int = 0
    grid_w: int = 0
    lm_h: int = 0
    lm_w: int = 0
    scale: float = 0.0
    flags: int = 0
    dtype: int = BF16

    def c(self):
        return _CParams(self.B, self.H, self.N, self.d, self.m, self.k, self.s, self.grid_h, self.grid_w,
                        self.lm_h, self.lm_w, float(self.scale), int(self.flags), int(self.dtype))


def lib():
    """The loaded libmita.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmita.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(_CParams)
        vp, sz, ip, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p
        L.mita_workspace_size.argtypes = [P]
        L.mita_workspace_size.restype = sz
        L.mita_landmarks.argtypes = [P, vp, fp, vp, sz, vp]
        L.mita_select.argtypes = [P, vp, vp, ip, ip, vp, sz, vp]
        L.mita_forward.argtypes = [P, vp, vp, vp, vp, ip, ip, fp, vp, sz, vp]
        L.mita_host_buffer_size.argtypes = [P]
        L.mita_host_buffer_size.restype = sz
        L.mita_forward_host.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
        L.mita_device_status.argtypes = [vp, vp]
        L.mita_status_string.argtypes = [ctypes.c_int]
        L.mita_status_string.restype = ctypes.c_char_p
        L.mita_last_error.argtypes = []
        L.mita_last_error.restype = ctypes.c_char_p
        L.mita_uses_tensor_cores.argtypes = [P]
        L.mita_backward_workspace_size.argtypes = [P]
        L.mita_backward_workspace_size.restype = sz
        L.mita_backward.argtypes = [P, vp, vp, vp, vp, ip, ip, vp, vp, vp, vp, sz, vp]
        L.mita_backward.restype = ctypes.c_int
        L.mita_forward_static.argtypes = [P, vp, vp, vp, vp, ip, vp]
        L.mita_forward_static.restype = ctypes.c_int
        L.mita_launch_count.argtypes = []
        L.mita_launch_count.restype = ctypes.c_longlong
        L.mita_profile_begin.argtypes = [ctypes.c_int]
        L.mita_profile_begin.restype = ctypes.c_int
        L.mita_profile_end.argtypes = [ctypes.c_char_p, sz, ctypes.POINTER(ctypes.c_double), ctypes.c_int]
        L.mita_profile_end.restype = ctypes.c_int
        for f in ("mita_landmarks", "mita_select", "mita_forward", "mita_forward_host", "mita_device_status",
                  "mita_uses_tensor_cores"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc):
    if rc:
        raise MitaError(rc, lib().mita_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def mita_workspace_size(p: Params) -> int:
    return int(lib().mita_workspace_size(ctypes.byref(p.c())))


def mita_host_buffer_size(p: Params) -> int:
    return int(lib().mita_host_buffer_size(ctypes.byref(p.c())))


def mita_uses_tensor_cores(p: Params) -> int:
    return int(lib().mita_uses_tensor_cores(ctypes.byref(p.c())))


def mita_launch_count() -> int:
    return int(lib().mita_launch_count())


def mita_profile_begin(max_marks: int):
    _check(lib().mita_profile_begin(int(max_marks)))


def mita_profile_end() -> dict:
    """Per-phase milliseconds summed over the calls since mita_profile_begin."""
    names = ctypes.create_string_buffer(4096)
    ms = (ctypes.c_double * 64)()
    n = lib().mita_profile_end(names, 4096, ms, 64)
    if n < 0:
        raise MitaError(4, "profile read failed")
    keys = names.value.decode().split("\n")[:n]
    return {k: ms[i] for i, k in enumerate(keys)}


def workspace(p: Params, device="cuda"):
    """A device workspace of the size ``p`` needs (torch uint8 tensor)."""
    import torch
    n = mita_workspace_size(p)
    if n == 0:
        raise MitaError(1, lib().mita_last_error().decode() or "invalid parameters")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mita_landmarks(p: Params, Q, Qt, ws, stream=None):
    _check(lib().mita_landmarks(ctypes.byref(p.c()), _ptr(Q), _ptr(Qt), _ptr(ws), ws.numel(), _stream(stream)))


def mita_select(p: Params, Q, K, idx, route, ws, stream=None):
    _check(lib().mita_select(ctypes.byref(p.c()), _ptr(Q), _ptr(K), _ptr(idx), _ptr(route), _ptr(ws), ws.numel(),
                             _stream(stream)))


def mita_forward(p: Params, Q, K, V, O, ws, idx_out=None, route_out=None, Vt_out=None, stream=None):
    _check(lib().mita_forward(ctypes.byref(p.c()), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(idx_out),
                              _ptr(route_out), _ptr(Vt_out), _ptr(ws), ws.numel(), _stream(stream)))


def mita_forward_static(p: Params, Q, K, V, O, status_out=None, stream=None):
    """The forward pass on the library's static device workspace (nothing is
    allocated): for callers that cannot allocate device memory. status_out is
    an optional int32 device tensor receiving the device status word. The
    call runs with Q's device current (the static area is per device)."""
    import torch
    with torch.cuda.device(Q.device):
        _check(lib().mita_forward_static(ctypes.byref(p.c()), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                         _ptr(status_out), _stream(stream)))


def mita_forward_host(p: Params, Q, K, V, O, dev, stream=None):
    """Q, K, V, O are host tensors (pinned for full copy speed); dev is a device
    buffer of mita_host_buffer_size(p) bytes."""
    _check(lib().mita_forward_host(ctypes.byref(p.c()), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dev), dev.numel(),
                                   _stream(stream)))


def mita_backward_workspace_size(p: Params) -> int:
    return int(lib().mita_backward_workspace_size(ctypes.byref(p.c())))


def mita_backward(p: Params, Q, K, V, dO, idx, route, dQ, dK, dV, ws, stream=None):
    _check(lib().mita_backward(ctypes.byref(p.c()), _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(idx), _ptr(route),
                               _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))


def backward(Q, K, V, dO, idx, route, m, k, s, scale=0.0, flags=0, ws=None):
    """Gradients (dQ, dK, dV) of sum(O * dO) for the forward pass with expert
    sets idx [B, H, m, k] and routes route [B, H, N, s] (torch CUDA tensors);
    the sets and routes are held fixed."""
    import torch
    p = params_for(Q, m, k, s, None, None, scale, flags)
    if ws is None:
        n = mita_backward_workspace_size(p)
        if n == 0:
            raise MitaError(2, lib().mita_last_error().decode() or "unsupported parameters")
        ws = torch.empty(n, dtype=torch.uint8, device=Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    mita_backward(p, Q, K, V, dO, idx, route, dQ, dK, dV, ws)
    mita_device_status(ws)
    return dQ, dK, dV


def mita_device_status(ws, stream=None):
    _check(lib().mita_device_status(_ptr(ws), _stream(stream)))


def params_for(Q, m, k, s, grid=None, lm=None, scale=0.0, flags=0) -> Params:
    """Params for torch tensors Q of shape [B, H, N, d]."""
    import torch
    B, H, N, d = Q.shape
    dt = {torch.float32: F32, torch.bfloat16: BF16}[Q.dtype]
    gh, gw = grid if grid else (0, 0)
    lh, lw = lm if lm else (0, 0)
    return Params(B, H, N, d, m, k, s, gh, gw, lh, lw, scale, flags, dt)


def forward(Q, K, V, m, k, s, grid=None, lm=None, scale=0.0, flags=0, return_sets=False, ws=None):
    """Convenience wrapper on torch CUDA tensors [B, H, N, d] (float32 or
    bfloat16). Returns O, or (O, idx, route, Vt) with ``return_sets``."""
    import torch
    p = params_for(Q, m, k, s, grid, lm, scale, flags)
    for t in (Q, K, V):
        if not t.is_cuda or not t.is_contiguous() or t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError("Q, K, V must be contiguous CUDA tensors of one shape and dtype")
    O = torch.empty_like(Q)
    if ws is None:
        ws = workspace(p, Q.device)
    if not return_sets:
        mita_forward(p, Q, K, V, O, ws)
        return O
    B, H, N, d = Q.shape
    idx = torch.empty((B, H, m, k), dtype=torch.int32, device=Q.device)
    route = torch.empty((B, H, N, s), dtype=torch.int32, device=Q.device)
    Vt = torch.empty((B, H, m, d), dtype=torch.float32, device=Q.device)
    mita_forward(p, Q, K, V, O, ws, idx, route, Vt)
    return O, idx, route, Vt
