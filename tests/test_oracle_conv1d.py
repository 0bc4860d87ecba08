"""Pins for the oracle's causal depthwise conv1d (the stage before the scan in a Mamba block):
a library routine, hand-derived closed forms and invariants.  CPU only."""
import numpy as np
import pytest
from scipy.special import expit

from selective_state_space_scan_gb300 import synth


def _inputs(seed, batch, L, Dm, K=4):
    g = synth.rng_for(seed, 9)
    x = g.standard_normal((batch, L, Dm), dtype=np.float32)
    w = (0.5 * g.standard_normal((Dm, K), dtype=np.float32)).astype(np.float32)
    bias = (0.1 * g.standard_normal(Dm, dtype=np.float32)).astype(np.float32)
    return x, w, bias


def test_conv1d_matches_numpy_correlate(oracle_mod):
    """Each (batch, channel) row is numpy's correlation of the zero-padded row with its weights."""
    x, w, bias = _inputs(1, 2, 37, 5)
    out, _ = oracle_mod.conv1d(x, w, bias, act=False)
    K = w.shape[1]
    for b in range(2):
        for d in range(5):
            padded = np.concatenate([np.zeros(K - 1), x[b, :, d].astype(np.float64)])
            ref = np.correlate(padded, w[d].astype(np.float64), mode="valid") + bias[d]
            np.testing.assert_allclose(out[b, :, d], ref, rtol=1e-13, atol=1e-14)


def test_conv1d_impulse_response(oracle_mod):
    """x = 1 at step t0, 0 elsewhere: out[t0 + j] = bias + w[K-1-j] for j < K, bias elsewhere.
    The newest sample meets the last weight (the orientation of the causal window)."""
    K, L, t0 = 4, 12, 5
    w = np.array([[1.0, 2.0, 3.0, 4.0], [-0.5, 0.25, 0.125, 8.0]], np.float32)
    bias = np.array([0.5, -1.0], np.float32)
    x = np.zeros((1, L, 2), np.float32)
    x[0, t0, :] = 1.0
    out, _ = oracle_mod.conv1d(x, w, bias, act=False)
    for d in range(2):
        expect = np.full(L, float(bias[d]))
        for j in range(K):
            expect[t0 + j] += float(w[d, K - 1 - j])
        np.testing.assert_array_equal(out[0, :, d], expect)


def test_conv1d_constant_input_and_left_edge(oracle_mod):
    """x = c everywhere: the first K-1 outputs see only the last t+1 weights (zero padding),
    later ones the whole sum."""
    K, L, c = 4, 9, 1.5
    w = np.array([[0.25, -1.0, 2.0, 0.5]], np.float32)
    x = np.full((1, L, 1), c, np.float32)
    out, win = oracle_mod.conv1d(x, w, None, act=False)
    for t in range(L):
        expect = c * float(w[0, max(0, K - 1 - t):].sum())
        assert out[0, t, 0] == pytest.approx(expect, rel=1e-15, abs=1e-15)
    np.testing.assert_array_equal(win[0, 0], [c] * (K - 1))


@pytest.mark.parametrize("k", [1, 2, 3, 11, 29])
def test_conv1d_split_composition(oracle_mod, k):
    """Convolving [0, k) then [k, L) from the window the first call left gives the one-call
    result, including pieces shorter than the window."""
    x, w, bias = _inputs(2, 2, 30, 4)
    win0 = synth.rng_for(3, 9).standard_normal((2, 4, 3))
    out, wout = oracle_mod.conv1d(x, w, bias, window=win0)
    o1, w1 = oracle_mod.conv1d(x[:, :k], w, bias, window=win0)
    o2, w2 = oracle_mod.conv1d(x[:, k:], w, bias, window=w1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), out, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(w2, wout, rtol=0, atol=0)


def test_conv1d_window_shift_for_short_calls(oracle_mod):
    """A one-step call (decode) shifts the window by one: [s0, s1, s2] -> [s1, s2, x0]."""
    w = np.ones((1, 4), np.float32)
    win = np.array([[[1.0, 2.0, 3.0]]])
    x = np.array([[[10.0]]], np.float32)
    out, wout = oracle_mod.conv1d(x, w, None, window=win, act=False)
    assert out[0, 0, 0] == 16.0
    np.testing.assert_array_equal(wout[0, 0], [2.0, 3.0, 10.0])
    x2 = np.array([[[10.0], [20.0]]], np.float32)
    _, wout2 = oracle_mod.conv1d(x2, w, None, window=win, act=False)
    np.testing.assert_array_equal(wout2[0, 0], [3.0, 10.0, 20.0])


def test_conv1d_silu(oracle_mod):
    x, w, bias = _inputs(4, 1, 20, 3)
    pre, _ = oracle_mod.conv1d(x, w, bias, act=False)
    out, _ = oracle_mod.conv1d(x, w, bias, act=True)
    np.testing.assert_allclose(out, pre * expit(pre), rtol=1e-14, atol=1e-300)
