"""ctypes front end of the fp64 MiTA oracle (``oracle/mita_oracle.c``).

Test infrastructure only: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its Python binding) never does, and shares no code with
it.

The oracle follows the MiTA forward pass step by step as described in
"MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of Top-k
Activations" (gist.science summaries; Dutch edition "Wiskundige Formulering"
for K* / V*, Arabic edition section 2 for the landmark queries, the shared
expert Vt = Atten(Qt, K, V) and the top-k index sets). Every array it takes is
float64 (inputs are widened exactly from their storage type before the call).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mita_oracle.c")
_LIB = os.path.join(_HERE, "libmita_oracle.so")
_lib = None


class MoParams(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int), ("d", ctypes.c_int), ("m", ctypes.c_int),
        ("k", ctypes.c_int), ("s", ctypes.c_int),
        ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int),
        ("lm_h", ctypes.c_int), ("lm_w", ctypes.c_int),
        ("scale", ctypes.c_double), ("no_shared", ctypes.c_int),
        ("causal", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        lib.mo_pool.argtypes = [ctypes.POINTER(MoParams), ctypes.c_int, dp, dp]
        lib.mo_scores.argtypes = [dp, ctypes.c_int, dp, ctypes.c_int, ctypes.c_int, dp]
        lib.mo_forward.argtypes = [ctypes.POINTER(MoParams), ctypes.c_int, dp, dp, dp,
                                   ctypes.c_int, ip, ip, ip, dp, dp, ip, ip, dp, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_uint64)]
        for f in (lib.mo_pool, lib.mo_scores, lib.mo_forward):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _params(N, d, m, k, s, grid=None, lm=None, scale=0.0, no_shared=False, causal=False):
    gh, gw = grid if grid else (1, N)
    lh, lw = lm if lm else (1, m)
    return MoParams(N, d, m, k, s, gh, gw, lh, lw, float(scale), int(bool(no_shared)), int(bool(causal)))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def pool(Q, m, grid=None, lm=None):
    """Landmark queries: Q [H, N, d] float64 -> Qt [H, m, d]."""
    Q = _f64(Q)
    H, N, d = Q.shape
    p = _params(N, d, m, 1, 1, grid, lm)
    Qt = np.empty((H, m, d))
    if _load().mo_pool(ctypes.byref(p), H, _dp(Q), _dp(Qt)):
        raise ValueError("oracle pool: bad parameters")
    return Qt


def scores(A, B):
    """Raw dot products S[i, j] = A[i] . B[j] in float64 (2-D inputs)."""
    A, B = _f64(A), _f64(B)
    S = np.empty((A.shape[0], B.shape[0]))
    _load().mo_scores(_dp(A), A.shape[0], _dp(B), B.shape[0], A.shape[1], _dp(S))
    return S


def forward(Q, K, V, m, k, s, grid=None, lm=None, scale=0.0, no_shared=False, q_ids=None,
            I_override=None, E_override=None, threads=None, causal=False):
    """MiTA forward for independent heads: Q, K, V [H, N, d] (float64).

    causal=True is this build's causal variant (1-D pooling only; the rules are
    in the header of mita_oracle.c): Vt_i over the keys of landmark i's prefix,
    a landmark's shared slot only once its bin is complete, routed keys up to
    the query's own position, zero output for a query with no slot.

    Returns a dict with Qt, Vt [H, m, d], I [H, m, k] (ascending), E [H, n_q, s]
    (descending routing score), O [H, n_q, d] and the multiply-add count.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    H, N, d = Q.shape
    p = _params(N, d, m, k, s, grid, lm, scale, no_shared, causal)
    if q_ids is None:
        n_q, qp = N, None
    else:
        q_ids = np.ascontiguousarray(q_ids, dtype=np.int32)
        n_q, qp = len(q_ids), q_ids
    Io = None if I_override is None else np.ascontiguousarray(I_override, dtype=np.int32)
    Eo = None if E_override is None else np.ascontiguousarray(E_override, dtype=np.int32)
    Qt = np.empty((H, m, d)); Vt = np.empty((H, m, d))
    I = np.empty((H, m, k), dtype=np.int32); E = np.empty((H, n_q, s), dtype=np.int32)
    O = np.empty((H, n_q, d))
    macs = ctypes.c_uint64(0)
    nth = threads if threads else (os.cpu_count() or 1)
    rc = _load().mo_forward(ctypes.byref(p), H, _dp(Q), _dp(K), _dp(V), n_q, _ip(qp), _ip(Io), _ip(Eo),
                            _dp(Qt), _dp(Vt), _ip(I), _ip(E), _dp(O), int(nth), ctypes.byref(macs))
    if rc == -1:
        raise ValueError("oracle forward: bad parameters")
    if rc:
        raise MemoryError("oracle forward: allocation failed")
    return {"Qt": Qt, "Vt": Vt, "I": I, "E": E, "O": O, "macs": int(macs.value)}
