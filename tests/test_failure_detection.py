"""Failure detection on the GPU without a fault: a bounded wait that nothing satisfies gives up
after its limit (about a second), records the timeout bit in the device error word and lets the
kernel finish; the context stays usable for the next call."""
import ctypes

import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import assert_fwd_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

WAIT_TIMEOUT_BIT = 1      # kErrWaitTimeout


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.device_error(clear=True)
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "publication-flag"])
def test_wait_that_never_completes_times_out_and_is_reported(kind):
    lib = ss.lib()
    lib.ss__wait_timeout_selftest.argtypes = [ctypes.c_int]
    lib.ss__wait_timeout_selftest.restype = ctypes.c_int
    assert lib.ss__wait_timeout_selftest(kind) == 1          # the kernel ran to its end
    assert ss.device_error(clear=True) & WAIT_TIMEOUT_BIT     # and said why it gave up
    assert ss.device_error() == 0                             # cleared
    # the context is still usable: a forward pass right after is correct and clean
    w = synth.config("tiny")
    a = w.arrays
    t = {k: (torch.from_numpy(v).cuda() if v is not None else None) for k, v in a.items()}
    y = ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"])
    torch.cuda.synchronize()
    ry, _, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"])
    assert_fwd_close("f32", y.cpu().numpy(), ry, mag, what="after the timeout")
    assert ss.device_error() == 0


def test_selftest_rejects_unknown_kind():
    lib = ss.lib()
    lib.ss__wait_timeout_selftest.argtypes = [ctypes.c_int]
    lib.ss__wait_timeout_selftest.restype = ctypes.c_int
    assert lib.ss__wait_timeout_selftest(7) == -1
