"""Parity checks of the CUDA path against the fp64 oracle.

The parity rules (expert sets, routes, outputs) for the
MiTA forward pass:

* Expert sets I_i: if the oracle's k-th and (k+1)-th raw scores differ by more
  than GAP, the CUDA set must equal the oracle's exactly; otherwise every
  CUDA-selected index must score within GAP of the oracle's k-th score. Sets
  must hold k distinct in-range indices in ascending order.
* Routes: the same rule on the routing scores q . qt_i with s in place of k,
  and the routes must be listed by non-increasing score (within GAP).
* Outputs (and Vt): the oracle recomputes them on the CUDA path's own index
  sets and routes; |gpu - oracle| <= atol + rtol * |oracle| element-wise with
  atol = rtol = 2e-2 for bf16 and 1e-4 for float32.
"""
import numpy as np

import oracle
from compressed_attention_adaptive_gb300 import synth

GAP = 1e-3
TOL = {"bf16": 2e-2, "f32": 1e-4}


def to_torch(a, dtype, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_torch(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_index_sets(got, S, k, what="I"):
    """got [rows, k] int; S [rows, n] oracle raw scores (float64)."""
    n = S.shape[1]
    exact = tol = 0
    for r in range(S.shape[0]):
        g = got[r]
        assert np.all((g >= 0) & (g < n)), "%s row %d: index out of range" % (what, r)
        assert len(np.unique(g)) == k, "%s row %d: repeated index" % (what, r)
        order = np.lexsort((np.arange(n), -S[r]))
        kth = S[r, order[k - 1]]
        nxt = S[r, order[k]] if k < n else -np.inf
        if kth - nxt > GAP:
            ref = np.sort(order[:k])
            assert np.array_equal(np.sort(g), ref), "%s row %d: set differs with gap %.3g" % (what, r, kth - nxt)
            exact += 1
        else:
            worst = S[r, g].min()
            assert worst >= kth - GAP, "%s row %d: index scores %.6g < kth %.6g - gap" % (what, r, worst, kth)
            tol += 1
    return exact, tol


def check_sorted_ascending(I):
    assert np.all(np.diff(I, axis=-1) > 0), "index sets must be strictly ascending"


def check_routes(E, R, s):
    """E [n_q, s]; R [n_q, m] oracle routing scores."""
    check_index_sets(np.sort(E, axis=1), R, s, what="route")
    sc = np.take_along_axis(R, E, axis=1)
    assert np.all(np.diff(sc, axis=1) <= GAP), "routes not listed by descending score"


def assert_close(got, ref, dtype, what):
    t = TOL[dtype]
    excess = np.abs(got - ref) - (t + t * np.abs(ref))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 0, "%s: |%.6g - %.6g| beyond tolerance at %s" % (what, got[i], ref[i], i)
    return float(np.abs(got - ref).max())


def run_gpu(w, Qn, Kn, Vn, flags=0, scale=0.0):
    """Runs mita_forward on storage arrays [B, H, N, d]; returns numpy results."""
    import torch
    import compressed_attention_adaptive_gb300 as mita
    Q, K, V = (to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
    grid = w.grid if w.grid else None
    p = mita.params_for(Q, w.m, w.k, w.s, grid, w.lm, scale, flags)
    ws = mita.workspace(p)
    O, idx, route, Vt = mita.forward(Q, K, V, w.m, w.k, w.s, grid=grid, lm=w.lm, scale=scale, flags=flags,
                                     return_sets=True, ws=ws)
    mita.mita_device_status(ws)  # raises on a device-side timeout or index error
    Qt = torch.empty((w.B, w.H, w.m, w.d), dtype=torch.float32, device=Q.device)
    mita.mita_landmarks(p, Q, Qt, ws)
    mita.mita_device_status(ws)
    return {"O": from_torch(O), "I": idx.cpu().numpy(), "E": route.cpu().numpy(), "Vt": from_torch(Vt),
            "Qt": from_torch(Qt)}


def check_heads(w, Qn, Kn, Vn, g, heads, q_ids=None, no_shared=False, scale=0.0):
    """Checks heads (flat ids) of the GPU result g against the oracle."""
    BH = w.B * w.H
    flat = lambda a: a.reshape((BH,) + a.shape[2:])
    f64 = lambda a: synth.widen(flat(a)[heads], w.dtype)
    Q, K, V = f64(Qn), f64(Kn), f64(Vn)
    gI, gE, gO, gVt, gQt = (flat(g[x])[heads] for x in ("I", "E", "O", "Vt", "Qt"))
    if q_ids is not None:
        gE, gO = gE[:, q_ids], gO[:, q_ids]
    ref = oracle.forward(Q, K, V, w.m, w.k, w.s, grid=w.grid, lm=w.lm, scale=scale, no_shared=no_shared,
                         q_ids=q_ids, I_override=gI, E_override=gE)
    rtol_qt = 1e-5 if w.dtype == "bf16" else 1e-6
    np.testing.assert_allclose(gQt, ref["Qt"], rtol=rtol_qt, atol=1e-6)
    stats = {"exact": 0, "tol": 0}
    for h in range(len(heads)):
        check_sorted_ascending(gI[h])
        e, t = check_index_sets(gI[h], oracle.scores(ref["Qt"][h], K[h]), w.k)
        stats["exact"] += e
        stats["tol"] += t
        qs = np.arange(w.N) if q_ids is None else np.asarray(q_ids)
        check_routes(gE[h], oracle.scores(Q[h][qs], ref["Qt"][h]), w.s)
    stats["Vt"] = assert_close(gVt, ref["Vt"], w.dtype, "Vt")
    stats["O"] = assert_close(gO, ref["O"], w.dtype, "O")
    return stats
