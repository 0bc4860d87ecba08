"""Calls on a stream other than torch's current one: the binding's cached workspace is
allocated and zero-filled on the call's stream, so the schedules that use it (balanced,
time split, the backward's checkpoints) give the same results there as on the default
stream, including when a larger call grows the cached buffer."""
import numpy as np
import pytest

import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import f32dev, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def _dev(w):
    a = w.arrays
    return dict(u=to_dev(a["u"], w.io), delta_raw=to_dev(a["delta_raw"], w.io), z=to_dev(a["z"], w.io),
                B=to_dev(a["B"], w.io), C=to_dev(a["C"], w.io), A_log=f32dev(a["A_log"]), D=f32dev(a["D"]),
                delta_bias=f32dev(a["delta_bias"]))


def _fwd(t, stream, batch, Dm, N):
    last = torch.empty((batch, Dm, N), device="cuda")
    y = ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                  last_state=last, stream=stream, workspace=True)
    return y, last


# (batch, L, Dm): many tiles (balanced schedule), then one row (time split), then a larger
# one-row call that grows the side stream's cached workspace
SHAPES = [(8, 256, 512), (1, 4096, 64), (1, 8192, 128)]


def test_forward_with_workspace_on_a_side_stream():
    side = torch.cuda.Stream()
    for i, (batch, L, Dm) in enumerate(SHAPES):
        w = synth.fwd_inputs(batch, L, Dm, 16, seed=80 + i)
        t = _dev(w)
        y0, l0 = _fwd(t, None, batch, Dm, 16)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            y1, l1 = _fwd(t, side, batch, Dm, 16)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        # same schedule and workspace size on both streams: bitwise equal
        assert np.array_equal(to_host(y0), to_host(y1)), (batch, L, Dm)
        assert np.array_equal(to_host(l0), to_host(l1)), (batch, L, Dm)


def test_backward_on_a_side_stream():
    side = torch.cuda.Stream()
    batch, L, Dm, N = 1, 4096, 64, 16          # few tiles: the backward's time split
    w = synth.fwd_inputs(batch, L, Dm, N, seed=90)
    t = _dev(w)
    dy = torch.randn((batch, L, Dm), device="cuda", generator=torch.Generator("cuda").manual_seed(90))

    def grads(stream):
        return ss.ss_bwd(dy, t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                         stream=stream)
    g0 = grads(None)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g1 = grads(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for k in ("du", "ddelta_raw", "dz", "dh0"):
        assert np.array_equal(to_host(g0[k]), to_host(g1[k])), k
    for k in ("dB", "dC", "dA_log", "dD", "ddelta_bias"):           # atomics: the order of the sums varies
        a, b = to_host(g0[k]).astype(np.float64), to_host(g1[k]).astype(np.float64)
        assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(a), k
