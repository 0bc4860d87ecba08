"""ss_fwd_static: the forward pass for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc, or must not: a host whose allocator owns all device
memory, a runtime that forbids allocation once started, or a plugin interface with no
allocation hook.  For them ss_fwd_static runs the balanced schedule of ss_fwd_ws on a fixed
workspace built into the library's device code, and allocates nothing.

This file is collected last so that a run that stops at the first failure has already run
every other test; it passes both on its own in a fresh process and after the others.
"""
import ctypes

import numpy as np
import pytest

import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import BF16_REL_L2, FP32_REL_L2, rel_l2, to_dev, f32dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SS_STATIC_WORKSPACE_BYTES = 1 << 20   # the fixed array's size, as declared in include/selscan.h


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def _static_fn():
    f = ss.lib().ss_fwd_static
    f.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_int64] * 4 + [ctypes.POINTER(ss.FwdStrides), ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _call(w, use_static):
    """One forward pass through the C ABI: ss_fwd_static or the existing ss_fwd."""
    a = w.arrays
    t = dict(u=to_dev(a["u"], w.io), delta_raw=to_dev(a["delta_raw"], w.io), z=to_dev(a["z"], w.io),
             B=to_dev(a["B"], w.io), C=to_dev(a["C"], w.io), A_log=f32dev(a["A_log"]), D=f32dev(a["D"]),
             bias=f32dev(a["delta_bias"]))
    y = torch.empty_like(t["u"])
    last = torch.empty((w.batch, w.Dm, w.N), device="cuda")
    u, dr, z, B, C = t["u"], t["delta_raw"], t["z"], t["B"], t["C"]
    s = ss.FwdStrides(ss.SS_BF16 if w.io == "bf16" else ss.SS_F32, u.stride(0), u.stride(1),
                      dr.stride(0), dr.stride(1), z.stride(0), z.stride(1), y.stride(0), y.stride(1),
                      B.stride(0), B.stride(1), C.stride(0), C.stride(1))
    args = (u.data_ptr(), dr.data_ptr(), t["bias"].data_ptr(), t["A_log"].data_ptr(), B.data_ptr(),
            C.data_ptr(), t["D"].data_ptr(), z.data_ptr(), y.data_ptr(), last.data_ptr(),
            w.batch, w.L, w.Dm, w.N, ctypes.byref(s), torch.cuda.current_stream().cuda_stream)
    st = _static_fn()(*args) if use_static else ss.lib().ss_fwd(*args)
    torch.cuda.synchronize()
    assert st == 0, ss.status_string(st)
    return to_host(y), to_host(last)


@pytest.mark.parametrize("name", ["mamba130m", "split", "bf16"])
def test_static_workspace_matches_ss_fwd_twice(name):
    """Two calls in a row (the second reuses the array the first left behind) agree with
    ss_fwd within the parity tolerance."""
    if name == "split":
        w = synth.fwd_inputs(6, 1000, 4096, 16, seed=31)       # ranges split tiles between CTAs
    elif name == "bf16":
        w = synth.fwd_inputs(8, 700, 1536, 16, io="bf16", seed=32)
    else:
        w = synth.config(name)
    io = ss.SS_BF16 if w.io == "bf16" else ss.SS_F32
    need = ss.lib().ss_fwd_workspace_size(w.batch, w.L, w.Dm, w.N, io)
    assert 0 < need <= SS_STATIC_WORKSPACE_BYTES                # the static path is really used
    y_ref, last_ref = _call(w, use_static=False)
    tol = BF16_REL_L2 if w.io == "bf16" else FP32_REL_L2
    for _ in range(2):
        y, last = _call(w, use_static=True)
        assert np.all(np.isfinite(y))
        assert rel_l2(y, y_ref) <= tol
        assert rel_l2(last, last_ref) <= FP32_REL_L2


def test_static_workspace_rejects_sizes_beyond_its_maximum():
    """A problem whose balanced schedule would need more than the fixed array (here the
    mamba-2.8b-shaped bf16 layer, about 1.2 MB of hand-over slots) is refused with
    SS_ERR_UNSUPPORTED before anything is enqueued."""
    batch, L, Dm, N = 4, 8192, 5120, 16
    need = ss.lib().ss_fwd_workspace_size(batch, L, Dm, N, ss.SS_BF16)
    assert need > SS_STATIC_WORKSPACE_BYTES
    s = ss.FwdStrides(ss.SS_BF16, L * Dm, Dm, L * Dm, Dm, L * Dm, Dm, L * Dm, Dm, L * N, N, L * N, N)
    dummy = torch.zeros(16, device="cuda")
    st = _static_fn()(*([dummy.data_ptr()] * 10), batch, L, Dm, N, ctypes.byref(s), None)
    assert st == 2                                              # SS_ERR_UNSUPPORTED
