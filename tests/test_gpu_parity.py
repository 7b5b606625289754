"""GPU parity of the MiTA forward pass (through the C ABI) against the oracle.

Small cases run every head and every query through the oracle; they span
several 128-row tiles with ragged tails, 1-D and 2-D pooling, both dtypes and
the degenerate settings. The full-size workloads are checked on sampled heads:
every landmark row's expert set, and every query's routes and output (the
vision, 32k and 131k workloads) or 1024 sampled queries (the sweep points).
"""
import math

import numpy as np
import pytest

from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

L = synth.WORKLOADS


def _case(w, seed=0, flags=0, heads=None, q_ids=None, scale=0.0):
    Qn, Kn, Vn = synth.make_inputs(w, seed=seed)
    g = parity.run_gpu(w, Qn, Kn, Vn, flags=flags, scale=scale)
    heads = list(range(w.BH)) if heads is None else heads
    return parity.check_heads(w, Qn, Kn, Vn, g, heads, q_ids=q_ids, no_shared=bool(flags & 1), scale=scale), g


SMALL = [
    L["fp32_n1024"],
    L["longctx_n32k"].with_(B=1, H=2, N=2048, m=16, k=200, s=2),
    L["longctx_n32k"].with_(B=2, H=1, N=1500, d=64, m=12, k=77, s=3),
    L["vision_128x128"].with_(B=1, H=2, N=1024, grid=(32, 32), lm=(4, 4), m=16, k=100, s=2),
    L["vision_128x128"].with_(B=1, H=1, N=30 * 20, grid=(30, 20), lm=(7, 3), m=21, k=64, s=4),
    L["n131k"].with_(B=1, H=1, N=4096, m=40, k=300, s=4),
    L["fp32_n1024"].with_(N=777, m=5, k=123, s=2, d=32),
    L["longctx_n32k"].with_(B=1, H=1, N=640, m=1, k=1, s=1),
    L["longctx_n32k"].with_(B=1, H=1, N=256, m=256, k=256, s=8),
    # experts cut into ragged 256-key sub-experts, and more than 256 landmarks
    # (the shared slots' own pass, also in ragged parts)
    L["n131k"].with_(B=1, H=1, N=4096, m=300, k=600, s=3),
    L["longctx_n32k"].with_(B=1, H=2, N=3000, d=64, m=200, k=520, s=2),
    # one head of the long-context shape: 128 key splits in the landmark pass
    # (the most the Vt combine sums), one sample chunk per CTA, a block per row
    # in the sample threshold, experts claimed in pieces
    L["longctx_n32k"].with_(B=1, H=1),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: "%s_N%d_d%d_m%d_k%d_s%d" % (w.dtype, w.N, w.d, w.m, w.k, w.s))
def test_small_cases_match_oracle(w):
    stats, _ = _case(w)
    assert stats["exact"] + stats["tol"] == w.BH * w.m


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_identity_no_shared_full_k_is_softmax_attention(dtype):
    import torch
    w = L["fp32_n1024"].with_(N=512, d=64, m=4, k=512, s=1, dtype=dtype)
    Qn, Kn, Vn = synth.make_inputs(w, seed=3)
    g = parity.run_gpu(w, Qn, Kn, Vn, flags=1)
    f = lambda a: torch.from_numpy(synth.widen(a, dtype)[0])
    ref = torch.nn.functional.scaled_dot_product_attention(f(Qn), f(Kn), f(Vn))[0].numpy()
    parity.assert_close(g["O"][0, 0], ref, dtype, "identity")


def test_explicit_scale():
    w = L["longctx_n32k"].with_(B=1, H=1, N=1024, m=8, k=128, s=2)
    _case(w, scale=0.05)


def test_simt_path_agrees_with_default_path():
    w = L["longctx_n32k"].with_(B=1, H=2, N=2048, m=32, k=256, s=2)
    Qn, Kn, Vn = synth.make_inputs(w, seed=5)
    a = parity.run_gpu(w, Qn, Kn, Vn)
    b = parity.run_gpu(w, Qn, Kn, Vn, flags=2)
    parity.assert_close(a["O"], b["O"], "bf16", "default vs CUDA-core path")
    parity.assert_close(a["Vt"], b["Vt"], "bf16", "Vt default vs CUDA-core path")


def test_repeat_calls_are_deterministic():
    w = L["longctx_n32k"].with_(B=1, H=2, N=2048, m=16, k=200, s=2)
    Qn, Kn, Vn = synth.make_inputs(w, seed=1)
    a = parity.run_gpu(w, Qn, Kn, Vn)
    b = parity.run_gpu(w, Qn, Kn, Vn)
    for x in ("O", "I", "E", "Vt"):
        np.testing.assert_array_equal(a[x], b[x])


def test_device_errors_and_statuses():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    w = L["longctx_n32k"].with_(B=1, H=1, N=512, m=4, k=16, s=1)
    Q = torch.zeros((1, 1, 512, 128), dtype=torch.bfloat16, device="cuda")
    p = mita.params_for(Q, 4, 16, 1)
    ws = mita.workspace(p)
    O = torch.empty_like(Q)
    with pytest.raises(mita.MitaError) as e:
        mita.mita_forward(p, Q, Q, Q, O, ws[: ws.numel() // 2])
    assert e.value.status == 3
    mita.mita_forward(p, Q, Q, Q, O, ws)
    mita.mita_device_status(ws)
    assert torch.isfinite(O.float()).all()


# ------------------------------------------------------------ full sizes

def _full(w, heads, n_q=None, seed=0):
    """Full-size workload on the GPU; the listed heads checked against the
    oracle on every landmark row, and on every query (n_q None) or on n_q
    sampled queries plus the first and the last."""
    Qn, Kn, Vn = synth.make_inputs(w, seed=seed)
    g = parity.run_gpu(w, Qn, Kn, Vn)
    q_ids = None
    if n_q is not None:
        rng = np.random.default_rng(seed)
        q_ids = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, n_q, replace=False)]))
    return parity.check_heads(w, Qn, Kn, Vn, g, heads, q_ids=q_ids)


def test_full_fp32_n1024():
    _case(L["fp32_n1024"])


def test_full_vision_128x128():
    _full(L["vision_128x128"], heads=[0, 37, 64, 95])


def test_full_longctx_n32k():
    _full(L["longctx_n32k"], heads=[0, 9, 22, 31])


@pytest.mark.slow
def test_full_n131k():
    _full(L["n131k"], heads=[3])


@pytest.mark.slow
@pytest.mark.parametrize("name", [w.name for w in synth.sweep_workloads()])
def test_full_sweep_points(name):
    _full(synth.get(name), heads=[7], n_q=1024)


# ---------------------------------------------- m and k raised at inference
# The pages note that m and k can be raised at inference time without
# retraining (Dutch edition, "Algorithmische Generalisatie"): the same fixed
# input as the benchmark's inference sweep, at the largest settings it times.

@pytest.mark.slow
@pytest.mark.parametrize("m,k", [(256, 1024), (512, 2048)])
def test_inference_raised_m_k(m, k):
    _full(L["longctx_n32k"].with_(B=1, H=16, m=m, k=k), heads=[5], n_q=1024)
