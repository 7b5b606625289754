"""Seeded synthetic inputs for the MiTA forward pass.

This module holds the workload definitions and the random input generators
that both the CUDA path and the oracle are fed from. It contains none of the
method's arithmetic: it only draws numbers, quantizes them once to the storage
dtype and widens stored values back to float64 exactly.

Every tensor of every (batch, head) is drawn from its own stream,
``numpy.random.default_rng(SeedSequence([seed, workload_id, b, h, tensor_id]))``,
so any single head can be regenerated on its own.

Storage: ``"f32"`` -> ``numpy.float32``; ``"bf16"`` -> ``numpy.uint16`` holding
bfloat16 bit patterns (round to nearest even from float32).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

try:  # scipy's FFT is faster and threaded; numpy's is the fallback
    import scipy.fft as _fft
except Exception:  # pragma: no cover
    _fft = np.fft


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int                 # workload id, part of every seed
    B: int
    H: int
    N: int
    d: int
    m: int
    k: int
    s: int
    dtype: str               # "f32" | "bf16"
    kind: str                # "iid" | "grf2d" | "clustered" | "ties"
    grid: tuple = None       # (grid_h, grid_w) for 2-D pooling
    lm: tuple = None         # (lm_h, lm_w) landmark grid for 2-D pooling
    k_centers: int = 64      # clustered: number of key centers
    v_kind: str = "clustered"  # clustered: "clustered" (own centers) or "iid"
    spread: float = 0.3      # clustered: within-cluster std
    q_noise: float = 0.5     # clustered: Q = K + q_noise * N(0, 1)
    length_scale: float = 8.0  # grf2d
    noise: float = 0.1       # grf2d: additive white-noise std
    zero_frac: float = 0.0   # ties: fraction of key rows set to zero (half of them -0.0)

    @property
    def BH(self):
        return self.B * self.H

    def with_(self, **kw):
        return dataclasses.replace(self, **kw)


# The five workloads: a small fp32 case, a vision-like 2-D grid, long context,
# a 131k-token case and the m x k x s sweep at 65k tokens.
WORKLOADS = {
    "fp32_n1024": Workload("fp32_n1024", 1, 1, 1, 1024, 64, 16, 64, 1, "f32", "iid"),
    "vision_128x128": Workload("vision_128x128", 2, 8, 12, 16384, 64, 64, 128, 2, "bf16", "grf2d",
                               grid=(128, 128), lm=(8, 8)),
    "longctx_n32k": Workload("longctx_n32k", 3, 2, 16, 32768, 128, 128, 256, 2, "bf16", "clustered"),
    "n131k": Workload("n131k", 4, 1, 8, 131072, 128, 256, 512, 4, "bf16", "clustered",
                      k_centers=256, v_kind="iid"),
}


def sweep_workloads():
    """The 27 points of the 65k-token sweep (m x k x s), clustered as longctx."""
    out = []
    for m in (32, 128, 512):
        for k in (64, 256, 1024):
            for s in (1, 2, 4):
                out.append(Workload("sweep_m%d_k%d_s%d" % (m, k, s), 5, 1, 16, 65536, 128, m, k, s,
                                    "bf16", "clustered"))
    return out


def get(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    for w in sweep_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


# ------------------------------------------------------------------ dtypes

def quantize(x, dtype: str):
    """float64/float32 array -> storage array (float32, or bf16 bits in uint16)."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x32
    if dtype != "bf16":
        raise ValueError(dtype)
    u = x32.view(np.uint32)
    # round to nearest, ties to even, on the upper 16 bits
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def widen(a, dtype: str):
    """Storage array -> float64, exactly."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    u = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def storage_np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


# -------------------------------------------------------------- generators

_TENSORS = {"Q": 0, "K": 1, "V": 2, "Z": 3}


def _rng(seed, w: Workload, b, h, tensor):
    return np.random.default_rng(np.random.SeedSequence([seed, w.wid, b, h, _TENSORS[tensor]]))


def _grf_kernel_hat(gh, gw, length_scale):
    """Spectrum of a periodic Gaussian kernel whose white-noise convolution has
    covariance length-scale ``length_scale``, normalized to unit variance."""
    sigma = length_scale / math.sqrt(2.0)

    def g1(n):
        r = np.minimum(np.arange(n), n - np.arange(n)).astype(np.float64)
        return np.exp(-(r ** 2) / (2 * sigma ** 2))

    g = np.outer(g1(gh), g1(gw))
    g /= math.sqrt((g ** 2).sum())
    return _fft.rfft2(g)


def _head(w: Workload, seed: int, b: int, h: int):
    """float32 Q, K, V [N, d] of one head before quantization."""
    N, d = w.N, w.d
    if w.kind == "iid":
        return tuple(_rng(seed, w, b, h, t).standard_normal((N, d), dtype=np.float32) for t in "QKV")
    if w.kind == "grf2d":
        gh, gw = w.grid
        khat = _grf_kernel_hat(gh, gw, w.length_scale)
        out = []
        for t in "QKV":
            rng = _rng(seed, w, b, h, t)
            white = rng.standard_normal((d, gh, gw))
            field = _fft.irfft2(_fft.rfft2(white) * khat, s=(gh, gw))
            field += w.noise * rng.standard_normal((d, gh, gw))
            out.append(np.ascontiguousarray(field.reshape(d, N).T, dtype=np.float32))
        return tuple(out)
    if w.kind == "clustered":
        rz = _rng(seed, w, b, h, "Z")
        z = rz.integers(0, w.k_centers, size=N)
        rk = _rng(seed, w, b, h, "K")
        ck = rk.standard_normal((w.k_centers, d), dtype=np.float32)
        K = ck[z] + np.float32(w.spread) * rk.standard_normal((N, d), dtype=np.float32)
        rv = _rng(seed, w, b, h, "V")
        if w.v_kind == "iid":
            V = rv.standard_normal((N, d), dtype=np.float32)
        else:
            cv = rv.standard_normal((w.k_centers, d), dtype=np.float32)
            V = cv[z] + np.float32(w.spread) * rv.standard_normal((N, d), dtype=np.float32)
        rq = _rng(seed, w, b, h, "Q")
        Q = K + np.float32(w.q_noise) * rq.standard_normal((N, d), dtype=np.float32)
        return Q, K, V
    if w.kind == "ties":
        # Small integers drawn from k_centers row patterns, so that raw scores
        # are exact in float32 and float64 and many of them are exactly equal.
        # Keys: pattern rows plus a zero_frac share of zero rows, half of them
        # -0.0. Queries: the first half of the 1-D pooling windows repeat a
        # period dividing the window, so their landmarks are identical (exact
        # routing ties); the rest are random pattern rows. With power-of-two
        # windows every landmark (a window mean) is exact too.
        rk = _rng(seed, w, b, h, "K")
        pat = rk.integers(-2, 3, size=(w.k_centers, d)).astype(np.float32)
        K = pat[rk.integers(0, w.k_centers, size=N)]
        nz = int(round(w.zero_frac * N))
        if nz:
            zr = rk.choice(N, nz, replace=False)
            K[zr] = 0.0
            K[zr[::2]] = -0.0
        rq = _rng(seed, w, b, h, "Q")
        qpat = rq.integers(-2, 3, size=(w.k_centers, d)).astype(np.float32)
        Q = qpat[rq.integers(0, w.k_centers, size=N)]
        win = N // w.m
        period = 4 if win % 4 == 0 and w.k_centers >= 4 else 1
        half = (w.m // 2) * win
        Q[:half] = qpat[np.arange(half) % period]
        V = _rng(seed, w, b, h, "V").standard_normal((N, d), dtype=np.float32)
        return Q, K, V
    raise ValueError(w.kind)


def make_head(w: Workload, seed: int, b: int, h: int):
    """Quantized (storage dtype) Q, K, V of one head, each [N, d]."""
    return tuple(quantize(x, w.dtype) for x in _head(w, seed, b, h))


def make_inputs(w: Workload, seed: int = 0, heads=None, threads: int = None):
    """Storage-dtype Q, K, V of shape [B, H, N, d] (or [len(heads), N, d] when
    ``heads`` lists flat head ids b*H + h)."""
    ids = list(range(w.BH)) if heads is None else list(heads)
    dt = storage_np_dtype(w.dtype)
    Q = np.empty((len(ids), w.N, w.d), dtype=dt)
    K = np.empty_like(Q)
    V = np.empty_like(Q)

    def one(i):
        bh = ids[i]
        Q[i], K[i], V[i] = make_head(w, seed, bh // w.H, bh % w.H)

    nth = threads or min(len(ids), os.cpu_count() or 1)
    if nth > 1:
        with ThreadPoolExecutor(nth) as ex:
            list(ex.map(one, range(len(ids))))
    else:
        for i in range(len(ids)):
            one(i)
    if heads is None:
        shape = (w.B, w.H, w.N, w.d)
        return Q.reshape(shape), K.reshape(shape), V.reshape(shape)
    return Q, K, V
