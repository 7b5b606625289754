"""Exact tie-breaking of the CUDA path: expert sets and routes on inputs whose
scores are exact in float32 and float64 and full of exact ties.

The top-k sets of "MiTA Attention: Efficient Fast-Weight Scaling via a Mixture
of Top-k Activations" (gist.science, Dutch edition "Kernconcepten" 3: the k
most activated key-value pairs per landmark) leave ties open; this library
breaks them towards the lower key index (and routing ties towards the lower
landmark index), with -0.0 equal to +0.0. The gap rule of the other parity
tests accepts any index within 1e-3 of the k-th score, so it cannot see the
tie rule. Here the inputs are small integers (keys from a few row patterns,
some rows +0.0 or -0.0; landmarks over power-of-two windows, half of them
identical), so every score the kernels compute is exact and the sets and
routes must equal the oracle's exactly, element for element.
"""
import numpy as np
import pytest

import oracle
from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu


def W(name, **kw):
    base = dict(name=name, wid=6, B=1, H=2, N=4096, d=128, m=32, k=256, s=2, dtype="bf16", kind="ties",
                k_centers=8, zero_frac=0.5)
    base.update(kw)
    return synth.Workload(**base)


TIES = [
    W("resident_zero_band", N=1024, m=16, k=256, s=2, zero_frac=0.6),  # the k-th score is 0 in half the rows
    W("resident", N=4096, m=32, k=256, s=2),
    W("resident_d64", N=2048, d=64, m=16, k=128, s=3, zero_frac=0.3),
    W("sub_experts_zero_band", N=4096, m=64, k=1024, s=3, zero_frac=0.4),  # four 256-key sub-experts
    W("route_m256", N=4096, m=256, k=128, s=8, zero_frac=0.2),
    W("route_chunked_m512", N=8192, m=512, k=64, s=4, k_centers=4, zero_frac=0.0),
    W("all_rows_equal", N=2048, m=16, k=100, s=2, k_centers=1, zero_frac=0.0),
    W("cuda_core_f32", N=1024, d=64, m=16, k=64, s=2, dtype="f32", zero_frac=0.7),
    W("longctx_32k", N=32768, m=128, k=256, s=2, zero_frac=0.5),
]


@pytest.mark.parametrize("w", TIES, ids=lambda w: w.name)
def test_ties_match_oracle_exactly(w):
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    g = parity.run_gpu(w, Qn, Kn, Vn)
    f = lambda a: synth.widen(a.reshape(w.BH, w.N, w.d), w.dtype)
    Q, K, V = f(Qn), f(Kn), f(Vn)
    ref = parity.oracle_parallel(Q, K, V, w)  # the oracle's own sets and routes
    gI = g["I"].reshape(w.BH, w.m, w.k)
    gE = g["E"].reshape(w.BH, w.N, w.s)
    np.testing.assert_array_equal(g["Qt"].reshape(w.BH, w.m, w.d), ref["Qt"])  # window means are exact
    for h in range(w.BH):
        S = oracle.scores(ref["Qt"][h], K[h])
        kth = np.sort(S, axis=1)[:, -w.k]
        # the inputs do what they are for: ties at the k-th score in most rows
        ties = (S == kth[:, None]).sum(axis=1) > 1
        assert ties.mean() > 0.5, "tie inputs produced too few ties"
        for r in range(w.m):
            assert np.array_equal(gI[h, r], ref["I"][h, r]), \
                "expert set %d of head %d differs (tie rule): gpu %s.. oracle %s.." % (
                    r, h, gI[h, r][:8], ref["I"][h, r][:8])
        bad = np.flatnonzero(~np.all(gE[h] == ref["E"][h], axis=1))
        assert len(bad) == 0, "route of query %d (head %d): gpu %s oracle %s" % (
            bad[0], h, gE[h, bad[0]], ref["E"][h, bad[0]])
    parity.assert_close(g["Vt"].reshape(w.BH, w.m, w.d), ref["Vt"], w.dtype, "ties %s Vt" % w.name)
    parity.assert_close(g["O"].reshape(w.BH, w.N, w.d), ref["O"], w.dtype, "ties %s O" % w.name)
