"""GPU parity of the causal variant against the oracle.

The pages describe no causal form of MiTA; this library's reading (1-D
pooling): the shared expert of landmark i attends to the keys of its prefix,
a query has landmark i's shared slot only once its bin is complete, routed
keys count only up to the query's own position, and a query left with no
slot gets a zero row. The oracle implements the same reading and is pinned
(tests/test_oracle_pins.py) against causal softmax attention and masked
attention built from library routines.
"""
import numpy as np
import pytest

from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

L = synth.WORKLOADS
CAUSAL = 4

CASES = [
    L["longctx_n32k"].with_(B=1, H=2, N=2048, m=16, k=200, s=2),
    L["longctx_n32k"].with_(B=1, H=2, N=4096, m=128, k=256, s=2),
    L["longctx_n32k"].with_(B=2, H=1, N=1500, d=64, m=12, k=77, s=3),   # bins not divisible, ragged tiles
    L["longctx_n32k"].with_(B=1, H=1, N=1024, m=8, k=16, s=1),          # early queries have no slot at all
    L["fp32_n1024"].with_(m=16, k=64, s=2),                              # CUDA-core path
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: "%s_N%d_d%d_m%d_k%d_s%d" % (w.dtype, w.N, w.d, w.m, w.k, w.s))
def test_causal_matches_oracle(w):
    Qn, Kn, Vn = synth.make_inputs(w, seed=2)
    g = parity.run_gpu(w, Qn, Kn, Vn, flags=CAUSAL)
    stats = parity.check_heads(w, Qn, Kn, Vn, g, list(range(w.BH)), causal=True, label="causal %s" % w.name)
    assert stats["exact"] + stats["tol"] == w.BH * w.m
    assert np.isfinite(g["O"]).all()
    if w.N == 1024 and w.m == 8:
        assert (np.abs(g["O"][0, 0, :20]).max(axis=-1) == 0).any()  # zero rows where no slot remains


def test_causal_full_longctx_n32k():
    w = L["longctx_n32k"].with_(B=1, H=2)
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    g = parity.run_gpu(w, Qn, Kn, Vn, flags=CAUSAL)
    parity.check_heads(w, Qn, Kn, Vn, g, [0, 1], causal=True, label="causal longctx N32768")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_causal_no_shared_full_k_is_causal_attention(dtype):
    # k = N, s = 1, shared slots off: causal softmax attention (CUDA-core path)
    import torch
    w = L["fp32_n1024"].with_(N=384, d=64, m=4, k=384, s=1, dtype=dtype)
    Qn, Kn, Vn = synth.make_inputs(w, seed=3)
    g = parity.run_gpu(w, Qn, Kn, Vn, flags=CAUSAL | 1 | 2)
    f = lambda a: torch.from_numpy(synth.widen(a, dtype)[0])
    ref = torch.nn.functional.scaled_dot_product_attention(f(Qn), f(Kn), f(Vn), is_causal=True)[0].numpy()
    parity.assert_close(g["O"][0, 0], ref, dtype, "causal identity %s" % dtype)


def test_causal_unsupported_shapes_are_rejected():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    Q = torch.zeros((1, 1, 2048, 128), dtype=torch.bfloat16, device="cuda")
    O = torch.empty_like(Q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p = mita.params_for(Q, 16, 512, 2, flags=CAUSAL)  # k > 256 on the tensor-core path
    with pytest.raises(mita.MitaError) as e:
        mita.mita_forward(p, Q, Q, Q, O, ws)
    assert e.value.status == 2, e.value  # MITA_ERR_UNSUPPORTED, before anything is enqueued
    p = mita.params_for(Q, 16, 512, 2, flags=CAUSAL | 2)  # the CUDA-core path runs it
    ws = mita.workspace(p)
    mita.mita_forward(p, Q, Q, Q, O, ws)
    mita.mita_device_status(ws)
