"""The single-launch time split of ss_fwd (no workspace): the CTAs that fold the time segments of
one channel tile form a thread-block cluster, fold their segments from a zero state, exchange the
(end state, Σ Δ) summaries through distributed shared memory, compose the state entering each
segment (the running prefix of "mamba-metal: Apple Silicon で Mamba を動かす", section
"チャンク間 running prefix", carried from cluster peer to cluster peer) and fold again from it.

Against the fp64 oracle on ragged lengths, both I/O types, with and without the gate and from an
initial state; at full size on the long-sequence workload (sampled rows); and the automatic choice.
"""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import assert_fwd_close, f32dev, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def _plan(w):
    f = ss.lib().ss__fwd_plan
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int32, ctypes.c_int, ctypes.c_char_p, ctypes.c_int]
    buf = ctypes.create_string_buffer(128)
    f(w.batch, w.L, w.Dm, w.N, ss.SS_BF16 if w.io == "bf16" else ss.SS_F32, 0, buf, 128)
    return buf.value.decode()


def _run(w, h0=None, force_cluster=True):
    lib = ss.lib()
    lib.ss__force_fwd_variant.argtypes = [ctypes.c_int] * 3
    a = w.arrays
    io = w.io
    last = torch.full((w.batch, w.Dm, w.N), float("nan"), device="cuda")
    if force_cluster:
        assert lib.ss__force_fwd_variant(2, 0, -1) == 0
    try:
        y = ss.ss_fwd(to_dev(a["u"], io), to_dev(a["delta_raw"], io), f32dev(a["delta_bias"]), f32dev(a["A_log"]),
                      to_dev(a["B"], io), to_dev(a["C"], io), f32dev(a["D"]), to_dev(a["z"], io), last_state=last,
                      workspace=False, h0=None if h0 is None else f32dev(h0))
        torch.cuda.synchronize()
    finally:
        lib.ss__force_fwd_variant(-1, 0, -1)
    return to_host(y), to_host(last)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [65, 130, 640, 1000, 4097])
def test_cluster_split_lengths(io, L):
    w = synth.fwd_inputs(1, L, 96, 16, io=io, seed=600 + L)
    y, last = _run(w)
    a = w.arrays
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"])
    assert_fwd_close(io, y, ry, mag, last, rl, what=f"cluster L={L} {io}")


def test_cluster_split_without_gate_and_from_h0():
    w = synth.fwd_inputs(2, 777, 64, 16, seed=610, with_z=False, with_D=False, with_bias=False)
    h0 = synth.initial_state(2, 64, 16, seed=611)
    y, last = _run(w, h0=h0)
    a = w.arrays
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"],
                                h0=h0.astype(np.float64))
    assert_fwd_close("f32", y, ry, mag, last, rl, what="cluster no gate, h0")


def test_cluster_split_partial_tile_and_one_chunk():
    """A tile that is not whole (Dm = 100), and a sequence of one chunk (the split does not apply:
    the segment kernel runs instead, same result)."""
    for L in (50, 300):
        w = synth.fwd_inputs(1, L, 100, 16, seed=620 + L)
        y, last = _run(w)
        a = w.arrays
        ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                    a["z"])
        assert_fwd_close("f32", y, ry, mag, last, rl, what=f"cluster Dm=100 L={L}")


def test_cluster_split_long_sequence_full_size():
    """The long-sequence workload (batch 1, L 32768, Dm 1536): ss_fwd without a workspace takes the
    cluster split automatically; every output of 24 sampled channels against the oracle."""
    w = synth.config("long32k")
    assert "cluster split" in _plan(w), _plan(w)
    y, last = _run(w, force_cluster=False)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(w.Dm, size=24, replace=False))
    a = w.arrays
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"],
                                rows=rows)
    assert_fwd_close("f32", y[0][:, rows].T, ry, mag, last[0][rows], rl, what="cluster long32k")
