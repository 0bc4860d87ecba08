"""ss_fwd_host (host-resident tensors, copies and scan overlapped over groups of batch rows)
against the fp64 oracle, and its argument checks."""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import assert_fwd_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def host(arr, io, pinned=True):
    if arr is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(arr, np.float32))
    if io == "bf16":
        t = t.to(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


def run(w, a, pinned=True, with_last=True, gate=True, params=True):
    io = w.io
    f32 = lambda x: None if x is None else host(x, "f32", pinned)
    last = torch.full((w.batch, w.Dm, w.N), float("nan")) if with_last else None
    if with_last and pinned:
        last = last.pin_memory()
    y = ss.ss_fwd_host(host(a["u"], io, pinned), host(a["delta_raw"], io, pinned),
                       f32(a["delta_bias"]) if params else None, f32(a["A_log"]), host(a["B"], io, pinned),
                       host(a["C"], io, pinned), f32(a["D"]) if params else None,
                       host(a["z"], io, pinned) if gate else None, last_state=last)
    torch.cuda.synchronize()
    return y.float().numpy(), (last.numpy() if with_last else None)


def check(w, a, what, **kw):
    y, last = run(w, a, **kw)
    gate, params = kw.get("gate", True), kw.get("params", True)
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"] if params else None, a["A_log"], a["B"],
                                a["C"], a["D"] if params else None, a["z"] if gate else None)
    assert_fwd_close(w.io, y, ry, mag, last, rl if last is not None else None, what=what)


@pytest.mark.parametrize("batch", [1, 3, 5, 8, 9])
def test_host_batch_groups(batch):
    """Row groups of ceil(batch / 8) rows: one group, ragged last groups, more groups than slots."""
    w = synth.fwd_inputs(batch, 300, 96, 16, seed=170 + batch)
    check(w, w.arrays, f"batch={batch}")


@pytest.mark.parametrize("L", [1, 63, 64, 65, 2049])
def test_host_lengths(L):
    w = synth.fwd_inputs(4, L, 64, 16, seed=180 + L)
    check(w, w.arrays, f"L={L}")


def test_host_bf16_and_optional_inputs():
    w = synth.fwd_inputs(6, 200, 64, 16, io="bf16", seed=190)
    check(w, w.arrays, "bf16")
    w = synth.fwd_inputs(6, 200, 40, 8, seed=191)
    check(w, w.arrays, "no gate, no D/bias, no last_state", gate=False, params=False, with_last=False)


def test_host_pageable_memory():
    w = synth.fwd_inputs(5, 150, 64, 16, seed=192)
    check(w, w.arrays, "pageable", pinned=False)


def test_host_full_size_130m_matches_device_call():
    """The 130m-shaped layer from host memory equals ss_fwd on device copies up to rounding
    (the groups may take another kernel variant), and meets the oracle's gates on sampled rows."""
    w = synth.config("mamba130m")
    a = w.arrays
    y, last = run(w, a)
    dev = {k: torch.from_numpy(v).cuda() for k, v in a.items() if v is not None}
    yd = ss.ss_fwd(dev["u"], dev["delta_raw"], dev["delta_bias"], dev["A_log"], dev["B"], dev["C"], dev["D"], dev["z"])
    torch.cuda.synchronize()
    yd = yd.cpu().numpy()
    assert np.linalg.norm(y - yd) / np.linalg.norm(yd) <= 1e-6
    rows = np.random.default_rng(5).choice(w.batch * w.Dm, 64, replace=False)
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"],
                                rows=rows)
    b, d = rows // w.Dm, rows % w.Dm
    assert_fwd_close("f32", y[b, :, d], ry, mag, last[b, d], rl, what="130m sampled rows")


def test_host_l0_zeroes_last_state():
    A_log = np.tile(np.log(np.arange(1, 17, dtype=np.float32)), (32, 1))
    last = torch.full((2, 32, 16), 7.0).pin_memory()
    z = np.zeros((2, 0, 32), np.float32)
    ss.ss_fwd_host(host(z, "f32"), host(z, "f32"), None, host(A_log, "f32"),
                   host(np.zeros((2, 0, 16), np.float32), "f32"), host(np.zeros((2, 0, 16), np.float32), "f32"),
                   last_state=last, y=torch.empty((2, 0, 32)).pin_memory())
    torch.cuda.synchronize()
    assert torch.count_nonzero(last) == 0


def test_host_rejects_device_pointers_and_small_workspace():
    w = synth.fwd_inputs(2, 64, 32, 16, seed=194)
    a = w.arrays
    lib = ss.lib()
    h = {k: host(v, "f32") for k, v in a.items() if v is not None}
    y = torch.empty((2, 64, 32)).pin_memory()
    need = lib.ss_fwd_host_workspace_size(2, 64, 32, 16, ss.SS_F32)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")

    def call(u_ptr, nbytes):
        return lib.ss_fwd_host(u_ptr, h["delta_raw"].data_ptr(), None, h["A_log"].data_ptr(), h["B"].data_ptr(),
                               h["C"].data_ptr(), None, None, y.data_ptr(), None, 2, 64, 32, 16, ss.SS_F32,
                               ws.data_ptr(), nbytes, None)
    u_dev = torch.from_numpy(a["u"]).cuda()
    assert call(u_dev.data_ptr(), need) == 1                  # a device pointer where host memory is expected
    assert call(h["u"].data_ptr(), need - 256) == 1           # workspace too small
    assert call(h["u"].data_ptr(), need) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("io,steps,batch", [("f32", 64, 9), ("bf16", 128, 3), ("f32", 1000, 2)])
def test_host_sequence_pieces(io, steps, batch):
    """The call cut into pieces of the sequence (forced here: 64 or 128 steps, against 300), each
    piece scanned from the state the previous one left on the device; two-row groups (batch 9)
    take strided copies.  With and without the gate and last_state."""
    f = ss.lib().ss__force_host_steps
    f.argtypes = [ctypes.c_int64]
    f.restype = ctypes.c_int64
    w = synth.fwd_inputs(batch, 300, 64, 16, io=io, seed=200 + steps + batch)
    f(steps)
    try:
        check(w, w.arrays, f"pieces of {steps} steps {io}")
        check(w, w.arrays, f"pieces of {steps} steps, no gate, no last_state", gate=False, with_last=False)
    finally:
        f(0)
