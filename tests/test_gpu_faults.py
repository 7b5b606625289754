"""Device-side failure detection, tested without a GPU fault.

Every wait of the tensor-core kernels on another role of the same CTA is
bounded. With MITA_TESTFLAG_STALL_PRODUCER, one CTA of the landmark pass
never loads its first key chunk and one CTA of the expert attention never
publishes its first query tile, and the waits give up after about a
millisecond. The call must report MITA_ERR_TIMEOUT through
mita_device_status (the wait ran out, the other roles left their loops), and
the next ordinary call on the same workspace must run clean and match the
oracle: the stalled CTAs let their copies and MMAs land and freed their tensor
memory, and nothing they left behind leaks into the next call.
"""
import numpy as np
import pytest

from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS["longctx_n32k"].with_(B=1, H=2, N=2048, m=16, k=200, s=2)


def _inputs():
    Qn, Kn, Vn = synth.make_inputs(W, seed=4)
    return (Qn, Kn, Vn), tuple(parity.to_torch(a, W.dtype) for a in (Qn, Kn, Vn))


def _normal_call_matches_oracle(mita, ws, host, dev):
    import torch
    Q, K, V = dev
    p = mita.params_for(Q, W.m, W.k, W.s)
    O = torch.empty_like(Q)
    idx = torch.empty((W.B, W.H, W.m, W.k), dtype=torch.int32, device=Q.device)
    route = torch.empty((W.B, W.H, W.N, W.s), dtype=torch.int32, device=Q.device)
    Vt = torch.empty((W.B, W.H, W.m, W.d), dtype=torch.float32, device=Q.device)
    mita.mita_forward(p, Q, K, V, O, ws, idx, route, Vt)
    mita.mita_device_status(ws)  # MITA_OK, or raises
    Qt = torch.empty((W.B, W.H, W.m, W.d), dtype=torch.float32, device=Q.device)
    mita.mita_landmarks(p, Q, Qt, ws)
    mita.mita_device_status(ws)
    g = {"O": parity.from_torch(O), "I": idx.cpu().numpy(), "E": route.cpu().numpy(),
         "Vt": parity.from_torch(Vt), "Qt": parity.from_torch(Qt)}
    parity.check_heads(W, *host, g, list(range(W.BH)), label="after a stalled call")


def test_stalled_forward_times_out_then_recovers():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    host, dev = _inputs()
    Q, K, V = dev
    p = mita.params_for(Q, W.m, W.k, W.s, flags=mita.TESTFLAG_STALL_PRODUCER)
    assert mita.mita_uses_tensor_cores(p) == 1
    ws = mita.workspace(p)
    O = torch.empty_like(Q)
    mita.mita_forward(p, Q, K, V, O, ws)  # enqueues; the timeout shows on the device
    with pytest.raises(mita.MitaError) as e:
        mita.mita_device_status(ws)
    assert e.value.status == 5, e.value  # MITA_ERR_TIMEOUT
    mita.mita_device_status(ws)  # reading the word cleared it
    _normal_call_matches_oracle(mita, ws, host, dev)


def test_stalled_landmark_pass_times_out_then_recovers():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    host, dev = _inputs()
    Q, K, V = dev
    p = mita.params_for(Q, W.m, W.k, W.s, flags=mita.TESTFLAG_STALL_PRODUCER)
    ws = mita.workspace(p)
    idx = torch.empty((W.B, W.H, W.m, W.k), dtype=torch.int32, device=Q.device)
    mita.mita_select(p, Q, K, idx, None, ws)  # landmark pass and top-k only
    with pytest.raises(mita.MitaError) as e:
        mita.mita_device_status(ws)
    assert e.value.status == 5, e.value
    _normal_call_matches_oracle(mita, ws, host, dev)


def test_stall_flag_is_accepted_but_inert_on_the_cuda_core_path():
    import torch
    import compressed_attention_adaptive_gb300 as mita
    w = synth.WORKLOADS["fp32_n1024"]
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    Q, K, V = (parity.to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
    p = mita.params_for(Q, w.m, w.k, w.s, flags=mita.TESTFLAG_STALL_PRODUCER)
    assert mita.mita_uses_tensor_cores(p) == 0
    ws = mita.workspace(p)
    O = torch.empty_like(Q)
    mita.mita_forward(p, Q, K, V, O, ws)
    mita.mita_device_status(ws)
    assert np.isfinite(parity.from_torch(O)).all()
