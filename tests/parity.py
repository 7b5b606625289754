"""Parity checks of the CUDA path against the fp64 oracle.

The parity rules (expert sets, routes, outputs) for the MiTA forward pass:

* Expert sets I_i: if the oracle's k-th and (k+1)-th raw scores differ by more
  than GAP, the CUDA set must equal the oracle's exactly; otherwise every
  CUDA-selected index must score within GAP of the oracle's k-th score. Sets
  must hold k distinct in-range indices in ascending order.
* Routes: the same rule on the routing scores q . qt_i with s in place of k,
  and the routes must be listed by non-increasing score (within GAP).
* Outputs (and Vt): the oracle recomputes them on the CUDA path's own index
  sets and routes; |gpu - oracle| <= atol + rtol * |oracle| element-wise with
  atol = rtol = 2e-2 for bf16 and 1e-4 for float32.

Every output comparison also records its headroom: the worst normalized
error |gpu - oracle| / (atol + rtol * |oracle|) (1.0 is the tolerance edge).
The suite prints the table at the end of the run (tests/conftest.py).
"""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

import oracle
from compressed_attention_adaptive_gb300 import synth

GAP = 1e-3
TOL = {"bf16": 2e-2, "f32": 1e-4}
REPORT = []  # (label, worst normalized error, max abs error, elements compared)


def to_torch(a, dtype, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_torch(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_index_sets(got, S, k, what="I"):
    """got [rows, k] int; S [rows, n] oracle raw scores (float64). Returns
    (rows checked by exact equality, rows checked by the gap allowance)."""
    got = np.asarray(got)
    rows, n = S.shape
    assert got.shape == (rows, k), "%s: shape %s, expected %s" % (what, got.shape, (rows, k))
    assert np.all((got >= 0) & (got < n)), "%s: index out of range" % what
    gs = np.sort(got, axis=1)
    assert np.all(np.diff(gs, axis=1) > 0), "%s: repeated index in a row" % what
    order = np.argsort(-S, axis=1, kind="stable")  # score descending, ties to the lower index
    kth = np.take_along_axis(S, order[:, k - 1:k], axis=1)[:, 0]
    nxt = np.take_along_axis(S, order[:, k:k + 1], axis=1)[:, 0] if k < n else np.full(rows, -np.inf)
    exact = kth - nxt > GAP
    ref = np.sort(order[:, :k], axis=1)
    bad = exact & ~np.all(gs == ref, axis=1)
    if bad.any():
        r = int(np.flatnonzero(bad)[0])
        raise AssertionError("%s row %d: set differs with gap %.3g" % (what, r, kth[r] - nxt[r]))
    worst = np.take_along_axis(S, got, axis=1).min(axis=1)
    bad = ~exact & (worst < kth - GAP)
    if bad.any():
        r = int(np.flatnonzero(bad)[0])
        raise AssertionError("%s row %d: index scores %.6g < kth %.6g - gap" % (what, r, worst[r], kth[r]))
    return int(exact.sum()), int((~exact).sum())


def check_sorted_ascending(I):
    assert np.all(np.diff(I, axis=-1) > 0), "index sets must be strictly ascending"


def check_routes(E, R, s):
    """E [n_q, s]; R [n_q, m] oracle routing scores."""
    check_index_sets(np.sort(E, axis=1), R, s, what="route")
    sc = np.take_along_axis(R, E, axis=1)
    assert np.all(np.diff(sc, axis=1) <= GAP), "routes not listed by descending score"


def assert_close(got, ref, dtype, what):
    """Element-wise tolerance check; returns the worst normalized error and
    records it (with the largest absolute error) in REPORT."""
    t = TOL[dtype]
    bound = t + t * np.abs(ref)
    diff = np.abs(got - ref)
    ratio = diff / bound
    i = np.unravel_index(np.argmax(ratio), ratio.shape)
    REPORT.append((what, float(ratio[i]), float(diff.max()), int(diff.size)))
    assert ratio[i] <= 1.0, "%s: |%.6g - %.6g| beyond tolerance at %s" % (what, got[i], ref[i], i)
    return float(ratio[i])


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


def oracle_parallel(Q, K, V, w, q_ids=None, I_override=None, E_override=None, no_shared=False, scale=0.0,
                    chunks=None, causal=False):
    """oracle.forward over heads Q, K, V [H, N, d], with each head's queries
    split into chunks that run on separate host threads (each chunk repeats the
    head's landmark pass; the oracle itself is unchanged). Returns the same
    dict as oracle.forward."""
    H = Q.shape[0]
    qs = np.arange(w.N) if q_ids is None else np.asarray(q_ids)
    cores = os.cpu_count() or 1
    if chunks is None:
        chunks = max(1, min(len(qs) // 256, -(-cores // H)))
    parts = np.array_split(np.arange(len(qs)), chunks)
    jobs = [(h, p) for h in range(H) for p in parts if len(p)]

    def one(job):
        h, p = job
        Io = None if I_override is None else I_override[h:h + 1]
        Eo = None if E_override is None else E_override[h:h + 1, p]
        return oracle.forward(Q[h:h + 1], K[h:h + 1], V[h:h + 1], w.m, w.k, w.s, grid=w.grid, lm=w.lm,
                              scale=scale, no_shared=no_shared, q_ids=qs[p], I_override=Io, E_override=Eo,
                              threads=1, causal=causal)

    with ThreadPoolExecutor(min(cores, len(jobs))) as ex:
        res = list(ex.map(one, jobs))
    out = {"Qt": np.empty((H, w.m, w.d)), "Vt": np.empty((H, w.m, w.d)), "I": np.empty((H, w.m, w.k), np.int32),
           "E": np.empty((H, len(qs), w.s), np.int32), "O": np.empty((H, len(qs), w.d)), "macs": 0}
    for (h, p), r in zip(jobs, res):
        for x in ("Qt", "Vt", "I"):
            out[x][h] = r[x][0]
        out["E"][h, p] = r["E"][0]
        out["O"][h, p] = r["O"][0]
        out["macs"] += r["macs"]
    return out


def check_heads(w, Qn, Kn, Vn, g, heads, q_ids=None, no_shared=False, scale=0.0, label=None, causal=False):
    """Checks heads (flat ids) of the GPU result g against the oracle."""
    BH = w.B * w.H
    flat = lambda a: a.reshape((BH,) + a.shape[2:])
    f64 = lambda a: synth.widen(flat(a)[heads], w.dtype)
    Q, K, V = f64(Qn), f64(Kn), f64(Vn)
    gI, gE, gO, gVt, gQt = (flat(g[x])[heads] for x in ("I", "E", "O", "Vt", "Qt"))
    if q_ids is not None:
        gE, gO = gE[:, q_ids], gO[:, q_ids]
    ref = oracle_parallel(Q, K, V, w, q_ids=q_ids, I_override=gI, E_override=gE, no_shared=no_shared, scale=scale,
                          causal=causal)
    rtol_qt = 1e-5 if w.dtype == "bf16" else 1e-6
    np.testing.assert_allclose(gQt, ref["Qt"], rtol=rtol_qt, atol=1e-6)
    stats = {"exact": 0, "tol": 0}
    qs = np.arange(w.N) if q_ids is None else np.asarray(q_ids)
    for h in range(len(heads)):
        check_sorted_ascending(gI[h])
        e, t = check_index_sets(gI[h], oracle.scores(ref["Qt"][h], K[h]), w.k)
        stats["exact"] += e
        stats["tol"] += t
        check_routes(gE[h], oracle.scores(Q[h][qs], ref["Qt"][h]), w.s)
    label = label or "%s N%d m%d k%d s%d" % (w.name, w.N, w.m, w.k, w.s)
    stats["Vt"] = assert_close(gVt, ref["Vt"], w.dtype, label + " Vt")
    stats["O"] = assert_close(gO, ref["O"], w.dtype, label + " O (%d heads x %d queries)" % (len(heads), len(qs)))
    return stats
