"""Chunk-length invariance of the forward scan on the GPU.

The sequence is folded chunk by chunk with the state carried across chunk boundaries ("mamba-metal:
Apple Silicon で Mamba を動かす", section "チャンク間 running prefix"), so where the chunks fall
must not change the result.  The library's lane kernels use 64-step chunks; test instantiations
of one configuration (fp32, 16 states at 4 lanes per channel, one CTA per 32-channel tile) at 16,
32 and 256 steps are selected through an internal hook.  At 256 steps a sequence of up to 256
steps is a single chunk: no carry is crossed.  Every chunk length is compared with the fp64
oracle, and with the 64-step kernel bit for bit (the fold visits the same steps in the same
order; only the staging of the tiles differs).
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

CHUNKS = [16, 32, 64, 256]


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def _run(w, chunk):
    lib = ss.lib()
    lib.ss__force_fwd_variant.argtypes = [ctypes.c_int] * 3
    lib.ss__force_chunk_steps.argtypes = [ctypes.c_int]
    lib.ss__force_chunk_steps.restype = ctypes.c_int
    a = w.arrays
    u, dr, z = to_dev(a["u"], w.io), to_dev(a["delta_raw"], w.io), to_dev(a["z"], w.io)
    Bm, Cm = to_dev(a["B"], w.io), to_dev(a["C"], w.io)
    last = torch.full((w.batch, w.Dm, w.N), float("nan"), device="cuda")
    assert lib.ss__force_fwd_variant(0, 4, 1) == 0
    assert lib.ss__force_chunk_steps(0 if chunk == 64 else chunk) >= 0
    try:
        y = ss.ss_fwd(u, dr, f32dev(a["delta_bias"]), f32dev(a["A_log"]), Bm, Cm, f32dev(a["D"]), z,
                      last_state=last, workspace=False)
        torch.cuda.synchronize()
    finally:
        lib.ss__force_chunk_steps(0)
        lib.ss__force_fwd_variant(-1, 0, -1)
    return to_host(y), to_host(last)


@pytest.mark.parametrize("L", [1, 31, 33, 200, 256, 1000, 2049])
def test_chunk_length_invariance(L):
    w = synth.fwd_inputs(2, L, 100, 16, seed=400 + L)
    a = w.arrays
    ref_y, ref_last, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"],
                                         a["D"], a["z"])
    base_y, base_last = _run(w, 64)
    for chunk in CHUNKS:
        y, last = _run(w, chunk)
        assert_fwd_close("f32", y, ref_y, mag, last, ref_last, what=f"chunk {chunk}, L={L}")
        np.testing.assert_array_equal(y, base_y, err_msg=f"chunk {chunk} vs 64, L={L}")
        np.testing.assert_array_equal(last, base_last, err_msg=f"chunk {chunk} vs 64, L={L}")


def test_chunk_override_refuses_other_configurations():
    """The test instantiations exist for one configuration only; anything else is refused, never
    silently run at the default chunk length."""
    lib = ss.lib()
    lib.ss__force_chunk_steps.argtypes = [ctypes.c_int]
    lib.ss__force_chunk_steps.restype = ctypes.c_int
    assert lib.ss__force_chunk_steps(48) == -1
    w = synth.fwd_inputs(1, 50, 64, 16, io="bf16", seed=499)
    a = w.arrays
    assert lib.ss__force_chunk_steps(32) >= 0
    try:
        with pytest.raises(ss.SelscanError):
            ss.ss_fwd(to_dev(a["u"], "bf16"), to_dev(a["delta_raw"], "bf16"), f32dev(a["delta_bias"]),
                      f32dev(a["A_log"]), to_dev(a["B"], "bf16"), to_dev(a["C"], "bf16"), f32dev(a["D"]),
                      to_dev(a["z"], "bf16"), workspace=False)
    finally:
        lib.ss__force_chunk_steps(0)
