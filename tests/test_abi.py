"""The C ABI library loads, exports every symbol include/mita.h declares and
validates arguments on the host (no GPU needed: nothing here launches)."""
import ctypes
import os
import re

import pytest

import compressed_attention_adaptive_gb300 as mita
from compressed_attention_adaptive_gb300 import build as mita_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mita_build.build()
    return mita.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(mita_\w+)\s*\(", src, re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"mita_forward", "mita_select", "mita_landmarks", "mita_workspace_size"} <= names
    for n in names:
        assert hasattr(lib, n), n


def _p(**kw):
    base = dict(B=1, H=2, N=1024, d=128, m=16, k=64, s=2)
    base.update(kw)
    return mita.Params(**base)


def test_workspace_size_and_validation(lib):
    assert mita.mita_workspace_size(_p()) > 0
    for bad in (dict(d=100), dict(m=0), dict(m=2048), dict(k=0), dict(k=4096), dict(s=0), dict(s=17),
                dict(s=9, m=64), dict(dtype=7), dict(flags=1 << 9), dict(grid_h=30, grid_w=30),
                dict(grid_h=32, grid_w=32, lm_h=3, lm_w=3), dict(scale=-1.0)):
        assert mita.mita_workspace_size(_p(**bad)) == 0, bad
        assert mita.mita_uses_tensor_cores(_p(**bad)) == -1, bad
    assert mita.mita_workspace_size(_p(grid_h=32, grid_w=32, lm_h=4, lm_w=4)) > 0


def test_host_side_errors_are_synchronous(lib):
    p = _p()
    rc = lib.mita_forward(ctypes.byref(p.c()), None, None, None, None, None, None, None, None, 0, None)
    assert rc == 1 and b"Q" in lib.mita_last_error()
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.mita_forward(ctypes.byref(p.c()), fake, fake, fake, fake, None, None, None, None, 0, None)
    assert rc == 3
    rc = lib.mita_forward(ctypes.byref(p.c()), fake, fake, fake, fake, None, None, None, ctypes.c_void_p(1 << 20 | 8),
                          1 << 40, None)
    assert rc == 3
    for s in range(7):
        assert lib.mita_status_string(s)
    assert mita.mita_host_buffer_size(p) > mita.mita_workspace_size(p)


def test_flag_values_match_the_header(lib):
    src = open(os.path.join(ROOT, "include", "mita.h")).read()
    assert re.search(r"MITA_FLAG_NO_SHARED\s*=\s*1u\s*<<\s*0\b", src) and mita.FLAG_NO_SHARED == 1
    assert re.search(r"MITA_FLAG_SIMT\s*=\s*1u\s*<<\s*1\b", src) and mita.FLAG_SIMT == 2
    assert re.search(r"#define\s+MITA_TESTFLAG_STALL_PRODUCER\s+\(1u\s*<<\s*31\)", src)
    assert mita.TESTFLAG_STALL_PRODUCER == 1 << 31
    # the fault-test flag is a valid flag (accepted on the host, like the others)
    assert mita.mita_workspace_size(_p(flags=mita.TESTFLAG_STALL_PRODUCER)) > 0


def test_causal_flag_validation(lib):
    C = mita.FLAG_CAUSAL
    assert mita.mita_workspace_size(_p(flags=C)) > 0                                      # resident shape
    assert mita.mita_workspace_size(_p(flags=C, grid_h=32, grid_w=32, lm_h=4, lm_w=4)) == 0  # 2-D pooling
    assert mita.mita_workspace_size(_p(flags=C, k=512)) == 0                              # unsupported on tcgen05
    assert mita.mita_workspace_size(_p(flags=C | mita.FLAG_SIMT, k=512)) > 0               # CUDA cores run it
    assert mita.mita_workspace_size(_p(flags=C, dtype=mita.F32, k=512)) > 0


def test_backward_workspace_and_validation(lib):
    assert mita.mita_backward_workspace_size(_p()) > 0
    assert mita.mita_backward_workspace_size(_p(flags=mita.FLAG_CAUSAL)) == 0                     # no causal backward
    assert mita.mita_backward_workspace_size(_p(grid_h=32, grid_w=32, lm_h=4, lm_w=4)) == 0       # 1-D pooling only
    p = _p()
    rc = lib.mita_backward(ctypes.byref(p.c()), *([None] * 9), None, 0, None)
    assert rc == 1 and b"aligned" in lib.mita_last_error()
