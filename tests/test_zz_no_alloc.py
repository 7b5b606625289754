"""mita_forward_static: the forward pass for callers that cannot allocate
device memory (the library brings a static device workspace).

Checked through the C ABI against mita_forward on a caller workspace, on two
calls in a row: the outputs must be identical (the static area keeps the
previous call's contents, so the second call shows nothing stale leaks in),
and the second call must leave the device's free memory unchanged. This file is collected last so a
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
    outs = []
    for seed in (0, 1):  # two calls in a row, different inputs
        Qn, Kn, Vn = synth.make_inputs(w, seed=seed)
        Q, K, V = (parity.to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
        p = mita.params_for(Q, w.m, w.k, w.s)
        ref = torch.empty_like(Q)
        ws = mita.workspace(p)
        mita.mita_forward(p, Q, K, V, ref, ws)
        got = torch.full_like(Q, float("nan"))
        st = torch.full((1,), -1, dtype=torch.int32, device=Q.device)
        torch.cuda.synchronize()
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        mita.mita_forward_static(p, Q, K, V, got, status_out=st)
        torch.cuda.synchronize()
        if seed == 1:
            # the first call on a device may load the library's device code;
            # after that a call allocates nothing, through torch or the driver
            assert torch.cuda.memory_allocated() == alloc0
            assert torch.cuda.mem_get_info()[0] == free0
        assert int(st.item()) == 0
        # same kernels, same inputs: the path is deterministic, so the outputs
        # are identical (nothing stale from the previous call leaks in)
        np.testing.assert_array_equal(parity.from_torch(got), parity.from_torch(ref))
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
