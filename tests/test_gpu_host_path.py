"""mita_forward_host (host buffers; the copies overlap the compute by groups
of heads) against mita_forward on the same inputs. The head counts cover
groups of one head, groups of two with the last one halved (16 heads: 7 x 2
+ 1 + 1) and of three with an uneven halving (24 heads: 7 x 3 + 2 + 1).

The two results differ only where the head count changes the key splits of
the shared-expert pass (a different summation order of its partials), so
they are compared at the bf16 output tolerance; the device status word of
the host path's workspace must read clean.
"""
import numpy as np
import pytest

from compressed_attention_adaptive_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [1, 3, 6, 16, 24])
def test_forward_host_matches_device(H):
    import torch
    import compressed_attention_adaptive_gb300 as mita
    w = synth.get("longctx_n32k").with_(B=1, H=H, N=4096)
    Qn, Kn, Vn = synth.make_inputs(w, seed=3)
    Q, K, V = (parity.to_torch(a, w.dtype) for a in (Qn, Kn, Vn))
    O = mita.forward(Q, K, V, w.m, w.k, w.s)
    p = mita.params_for(Q, w.m, w.k, w.s)
    hb = [torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).pin_memory() for a in (Qn, Kn, Vn)]
    hO = torch.full_like(hb[0], 0xFF).pin_memory()  # NaN bit patterns until written
    buf = torch.empty(mita.mita_host_buffer_size(p), dtype=torch.uint8, device="cuda")
    mita.mita_forward_host(p, hb[0], hb[1], hb[2], hO, buf)
    torch.cuda.synchronize()
    t = (hb[0].numel() + 1023) // 1024 * 1024  # Q, K, V, O, then the workspace
    mita.mita_device_status(buf[4 * t:])
    got = parity.from_torch(hO.view(torch.bfloat16).reshape(O.shape))
    ref = parity.from_torch(O)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=2e-2, atol=2e-2)
