"""GPU parity of the backward pass against the fp64 oracle backward.

The pages print no backward pass; oracle/backward.py is the chain rule through
the forward's steps with the expert sets and routes held fixed, pinned against
finite differences of the forward oracle (tests/test_oracle_pins.py). Here the
CUDA backward runs on the sets and routes of the CUDA forward, and the oracle
backward on the same sets and routes; dQ, dK, dV must agree element-wise
within atol = rtol = 2e-2 (bf16 storage) or 1e-4 (float32).
"""
import numpy as np
import pytest

from oracle import backward as obwd
from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

L = synth.WORKLOADS

CASES = [
    (L["fp32_n1024"].with_(N=512, m=8, k=64, s=2), 0),
    (L["longctx_n32k"].with_(B=1, H=2, N=1024, m=16, k=100, s=2), 0),
    (L["longctx_n32k"].with_(B=2, H=1, N=600, d=64, m=7, k=33, s=3), 0),   # bins not divisible
    (L["longctx_n32k"].with_(B=1, H=1, N=256, d=64, m=4, k=256, s=1), 1),  # shared slots off, every key
]


@pytest.mark.parametrize("w,flags", CASES, ids=lambda x: str(x) if isinstance(x, int) else "%s_N%d_d%d_m%d_k%d_s%d" % (
    x.dtype, x.N, x.d, x.m, x.k, x.s))
def test_backward_matches_oracle(w, flags):
    import torch
    import compressed_attention_adaptive_gb300 as mita
    Qn, Kn, Vn = synth.make_inputs(w, seed=5)
    Q, K, V = (parity.to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
    rng = np.random.default_rng(11)
    dOn = synth.quantize(rng.standard_normal(Qn.shape), w.dtype)
    dO = parity.to_torch(dOn, w.dtype)
    O, idx, route, Vt = mita.forward(Q, K, V, w.m, w.k, w.s, flags=flags, return_sets=True)
    dQ, dK, dV = mita.backward(Q, K, V, dO, idx, route, w.m, w.k, w.s, flags=flags)
    torch.cuda.synchronize()
    f = lambda a: synth.widen(a.reshape(w.BH, w.N, w.d), w.dtype)
    ref = obwd.backward(f(Qn), f(Kn), f(Vn), f(dOn), idx.cpu().numpy().reshape(w.BH, w.m, w.k),
                        route.cpu().numpy().reshape(w.BH, w.N, w.s), no_shared=bool(flags & 1))
    for name, got, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        parity.assert_close(parity.from_torch(got).reshape(w.BH, w.N, w.d), r, w.dtype,
                            "backward %s %s N%d" % (name, w.dtype, w.N))
