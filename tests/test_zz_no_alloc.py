"""mita_forward_static: the forward pass for callers that cannot allocate
device memory (the library brings a static device workspace).

Checked through the C ABI against mita_forward on a caller workspace, on two
calls in a row (the static area keeps the previous call's contents, so the
second call shows nothing stale leaks in). This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    synth.WORKLOADS["fp32_n1024"],  # CUDA-core path
    synth.WORKLOADS["longctx_n32k"].with_(B=1, H=2, N=2048, m=16, k=200, s=2),  # tensor-core path
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: "%s_N%d" % (w.dtype, w.N))
def test_static_workspace_matches_caller_workspace(w):
    import torch
    import compressed_attention_adaptive_gb300 as mita
    p_args = None
    outs = []
    for seed in (0, 1):  # two calls in a row, different inputs
        Qn, Kn, Vn = synth.make_inputs(w, seed=seed)
        Q, K, V = (parity.to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
        p = mita.params_for(Q, w.m, w.k, w.s)
        ref = torch.empty_like(Q)
        ws = mita.workspace(p)
        mita.mita_forward(p, Q, K, V, ref, ws)
        got = torch.empty_like(Q)
        st = torch.full((1,), -1, dtype=torch.int32, device=Q.device)
        mita.mita_forward_static(p, Q, K, V, got, status_out=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        parity.assert_close(parity.from_torch(got), parity.from_torch(ref), w.dtype, "static vs caller workspace")
        outs.append(parity.from_torch(got))
    assert not np.array_equal(outs[0], outs[1])


def test_static_workspace_rejects_oversized_problems():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    w = synth.WORKLOADS["longctx_n32k"]
    p = mita.Params(w.B, w.H, w.N, w.d, w.m, w.k, w.s)
    assert mita.mita_workspace_size(p) > (64 << 20)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mita.MitaError) as e:
        mita.mita_forward_static(p, x, x, x, x)
    assert e.value.status == 2
