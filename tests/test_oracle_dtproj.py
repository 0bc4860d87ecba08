"""Pins for the oracle's forward scan with the low-rank time-step projection folded in
(delta_raw = dt_low · W_dt^T): against the plain forward oracle fed the projection computed by
numpy's matmul, exactly where that projection is exactly representable, and to fp32 rounding
elsewhere.  CPU only."""
import numpy as np
import pytest

from selective_state_space_scan_gb300 import synth


def _dyadic(g, shape, lo, hi, step):
    return (g.integers(int(lo / step), int(hi / step) + 1, size=shape) * step).astype(np.float32)


def _problem(seed, batch=2, L=23, Dm=5, N=4):
    a = synth.fwd_inputs(batch, L, Dm, N, seed=seed).arrays
    g = np.random.default_rng(seed + 1000)
    return a, g


def test_dtproj_exact_projection_matches_plain_forward(oracle_mod):
    """dt_low and W on a 2^-4 grid in [-2, 2], R = 8: every product is a multiple of 2^-8 and the
    sums stay below 2^5, so numpy's fp64 matmul, rounded to fp32, is exact; both oracles then see
    the same time steps and agree bit for bit."""
    a, g = _problem(21)
    batch, L, Dm = a["u"].shape
    R = 8
    dt_low = _dyadic(g, (batch, L, R), -2, 2, 1 / 16)
    W = _dyadic(g, (Dm, R), -2, 2, 1 / 16)
    delta_raw = (dt_low.astype(np.float64) @ W.T.astype(np.float64)).astype(np.float32)
    assert np.array_equal(delta_raw.astype(np.float64), dt_low.astype(np.float64) @ W.T.astype(np.float64))
    y0, l0, m0 = oracle_mod.ss_fwd(a["u"], delta_raw, a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"])
    y1, l1, m1 = oracle_mod.ss_fwd_dtproj(a["u"], dt_low, W, a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                          a["z"])
    np.testing.assert_array_equal(y1, y0)
    np.testing.assert_array_equal(l1, l0)
    np.testing.assert_array_equal(m1, m0)


@pytest.mark.parametrize("R", [1, 4, 48])
def test_dtproj_general_projection_to_fp32_rounding(oracle_mod, R):
    """Normal dt_low, W: the plain oracle fed the fp32-rounded projection differs only by that
    rounding (relative 6e-8 in delta_raw)."""
    a, g = _problem(22 + R)
    batch, L, Dm = a["u"].shape
    dt_low = (0.3 * g.standard_normal((batch, L, R))).astype(np.float32)
    W = (g.standard_normal((Dm, R)) / np.sqrt(R)).astype(np.float32)
    delta_raw = (dt_low.astype(np.float64) @ W.T.astype(np.float64)).astype(np.float32)
    y0, l0, _ = oracle_mod.ss_fwd(a["u"], delta_raw, a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"])
    y1, l1, _ = oracle_mod.ss_fwd_dtproj(a["u"], dt_low, W, a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                         a["z"])
    np.testing.assert_allclose(y1, y0, rtol=1e-6, atol=1e-6 * np.abs(y0).max())
    np.testing.assert_allclose(l1, l0, rtol=1e-6, atol=1e-6 * np.abs(l0).max())
