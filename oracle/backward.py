"""fp64 backward pass of the MiTA forward -- part of the ORACLE.

Test infrastructure only, like the rest of ``oracle/``: the test suite and the
benchmark's CPU legs may use it; the product path never does, and shares no
code with it.

The pages describe the forward pass of "MiTA Attention: Efficient Fast-Weight
Scaling via a Mixture of Top-k Activations" (gist.science summaries: Arabic
edition section 2 for the landmarks, the shared expert and the expert sets;
Dutch edition "Wiskundige Formulering" for K* / V*) and report its training
speed, but print no backward pass. The gradient here is the plain chain rule
through the forward's steps, with the expert sets I and the routes E held
fixed (a top-k choice is piecewise constant: it has no gradient):

  output     O_t = sum_u P_tu val_u,  P_t = softmax_u(tau q_t . key_u) over the
             slots u of query t (the m shared slots (key Qt_i, value Vt_i),
             then the k keys of each routed expert)
  shared     Vt_i = sum_j A_ij v_j,   A_i = softmax_j(tau Qt_i . k_j)
  landmarks  Qt_i = mean of q_t over bin i

Backward, with dO given (D_t = dO_t . O_t, dZ_tu = P_tu (dO_t . val_u - D_t)):
  dq_t   += tau sum_u dZ_tu key_u
  shared slot i:  dQt_i += tau sum_t dZ_ti q_t,   dVt_i += sum_t P_ti dO_t
  routed key j:   dk_j  += tau dZ_tu q_t,         dv_j  += P_tu dO_t   (per slot)
  shared expert:  dS_ij = A_ij (dVt_i . v_j - dVt_i . Vt_i)
                  dQt_i += tau sum_j dS_ij k_j,  dk_j += tau sum_i dS_ij Qt_i,
                  dv_j  += sum_i A_ij dVt_i
  landmarks:      dq_t  += dQt_i / |bin_i| for each bin i holding t

Plain numpy, one head at a time, slot by slot; nothing is fused or blocked
beyond what these formulas state.
"""
from __future__ import annotations

import math

import numpy as np


def _bins(N, m):
    """1-D adaptive-average-pooling bins [floor(iN/m), ceil((i+1)N/m))."""
    return [(i * N // m, -(-(i + 1) * N // m)) for i in range(m)]


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def backward_head(Q, K, V, dO, I, E, scale=0.0, no_shared=False):
    """One head: Q, K, V, dO [N, d] float64; I [m, k], E [N, s] int (the
    forward's expert sets and routes). Returns dQ, dK, dV [N, d] float64."""
    N, d = Q.shape
    m = I.shape[0]
    tau = scale if scale > 0 else 1.0 / math.sqrt(d)
    bins = _bins(N, m)
    # forward quantities the chain rule needs
    Qt = np.stack([Q[lo:hi].mean(axis=0) for lo, hi in bins])          # [m, d]
    A = np.stack([_softmax(tau * (K @ Qt[i])) for i in range(m)])       # [m, N]
    Vt = A @ V                                                          # [m, d]
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dQt = np.zeros_like(Qt)
    dVt = np.zeros_like(Vt)
    for t in range(N):
        q = Q[t]
        keys, vals, kind, idx = [], [], [], []
        if not no_shared:
            for i in range(m):
                keys.append(Qt[i]); vals.append(Vt[i]); kind.append(0); idx.append(i)
        for e in E[t]:
            for j in I[e]:
                keys.append(K[j]); vals.append(V[j]); kind.append(1); idx.append(j)
        keys = np.array(keys); vals = np.array(vals)
        P = _softmax(tau * (keys @ q))
        O = P @ vals
        dP = vals @ dO[t]
        Dt = dO[t] @ O
        dZ = P * (dP - Dt)
        dQ[t] += tau * (dZ @ keys)
        for u in range(len(P)):
            if kind[u] == 0:
                dQt[idx[u]] += tau * dZ[u] * q
                dVt[idx[u]] += P[u] * dO[t]
            else:
                dK[idx[u]] += tau * dZ[u] * q
                dV[idx[u]] += P[u] * dO[t]
    if not no_shared:
        # shared expert Vt = A V with A = softmax(tau Qt K^T)
        dA = dVt @ V.T                                                  # [m, N]
        dS = A * (dA - np.sum(dVt * Vt, axis=1, keepdims=True))
        dQt += tau * (dS @ K)
        dK += tau * (dS.T @ Qt)
        dV += A.T @ dVt
        # landmarks: each query of bin i gets dQt_i / |bin_i|
        for i, (lo, hi) in enumerate(bins):
            dQ[lo:hi] += dQt[i] / (hi - lo)
    return dQ, dK, dV


def backward(Q, K, V, dO, I, E, scale=0.0, no_shared=False):
    """Independent heads: Q, K, V, dO [H, N, d]; I [H, m, k]; E [H, N, s]."""
    out = [backward_head(np.asarray(Q[h], np.float64), np.asarray(K[h], np.float64), np.asarray(V[h], np.float64),
                         np.asarray(dO[h], np.float64), np.asarray(I[h]), np.asarray(E[h]), scale, no_shared)
           for h in range(Q.shape[0])]
    return tuple(np.stack([o[c] for o in out]) for c in range(3))
