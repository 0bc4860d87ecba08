"""Pins for the oracle's backward scan: central finite differences of the (separately pinned)
forward oracle, and a closed form.  Inputs are multiples of 2^-8 and the step is 2^-12, so
every perturbed float input is exact and the difference quotient carries only its O(eps^2)
truncation error.  CPU only."""
import numpy as np
import pytest

from selective_state_space_scan_gb300 import synth

EPS = 2.0 ** -12


def _dyadic(g, shape, scale, lo=None):
    v = np.round(g.standard_normal(shape) * scale * 256) / 256
    if lo is not None:
        v = np.maximum(v, lo)
    return v.astype(np.float32)


def _problem(seed, batch=1, L=5, Dm=2, N=3, gate=True):
    g = synth.rng_for(seed, 11)
    a = dict(u=_dyadic(g, (batch, L, Dm), 1.0), delta_raw=_dyadic(g, (batch, L, Dm), 0.7),
             z=_dyadic(g, (batch, L, Dm), 1.0) if gate else None,
             B=_dyadic(g, (batch, L, N), 1.0), C=_dyadic(g, (batch, L, N), 1.0),
             A_log=_dyadic(g, (Dm, N), 0.5), D=_dyadic(g, (Dm,), 1.0), delta_bias=_dyadic(g, (Dm,), 0.3))
    h0 = _dyadic(g, (batch, Dm, N), 0.5).astype(np.float64)
    dy = _dyadic(g, (batch, L, Dm), 1.0)
    dlast = _dyadic(g, (batch, Dm, N), 1.0).astype(np.float64)
    return a, h0, dy, dlast


def _objective(oracle_mod, a, h0, dy, dlast):
    y, last, _ = oracle_mod.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                   a["z"], h0=h0)
    return float(np.sum(dy.astype(np.float64) * y) + np.sum(dlast * last))


@pytest.mark.parametrize("gate", [True, False], ids=["gate", "no_gate"])
def test_bwd_matches_finite_differences(oracle_mod, gate):
    a, h0, dy, dlast = _problem(3, gate=gate)
    grads = oracle_mod.ss_bwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                              a["z"], dy, h0=h0, dlast=dlast)
    names = {"u": "du", "delta_raw": "ddelta_raw", "B": "dB", "C": "dC", "A_log": "dA_log", "D": "dD",
             "delta_bias": "ddelta_bias"}
    if gate:
        names["z"] = "dz"
    for key, gname in names.items():
        fd = np.zeros(a[key].shape)
        for idx in np.ndindex(*a[key].shape):
            for sgn in (1, -1):
                b = dict(a)
                b[key] = a[key].copy()
                b[key][idx] = np.float32(a[key][idx] + sgn * EPS)
                assert float(b[key][idx]) == float(a[key][idx]) + sgn * EPS    # exact perturbation
                fd[idx] += sgn * _objective(oracle_mod, b, h0, dy, dlast)
        fd /= 2 * EPS
        scale = np.max(np.abs(fd)) + 1e-30
        np.testing.assert_allclose(grads[gname], fd, rtol=2e-6, atol=2e-6 * scale, err_msg=gname)
    # the initial state (double)
    fd = np.zeros(h0.shape)
    for idx in np.ndindex(*h0.shape):
        for sgn in (1, -1):
            hp = h0.copy()
            hp[idx] += sgn * EPS
            fd[idx] += sgn * _objective(oracle_mod, a, hp, dy, dlast)
    fd /= 2 * EPS
    np.testing.assert_allclose(grads["dh0"], fd, rtol=2e-6, atol=2e-6 * (np.max(np.abs(fd)) + 1e-30))


def test_bwd_A_to_zero_closed_form(oracle_mod):
    """A -> 0 and no gate: y_t = sum_n C_t,n sum_{s<=t} Delta_s B_s,n u_s + D u_t, so
    du_s = D dy_s + Delta_s sum_n B_s,n sum_{t>=s} dy_t C_t,n (a reverse cumulative sum)."""
    a, _, dy, _ = _problem(4, batch=2, L=17, Dm=3, N=4, gate=False)
    a["A_log"] = np.full_like(a["A_log"], -40.0)
    grads = oracle_mod.ss_bwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                              None, dy)
    dlt = np.logaddexp(0.0, a["delta_raw"].astype(np.float64) + a["delta_bias"][None, None, :])
    Cd = a["C"].astype(np.float64)
    # rev[b, s, d, n] = sum_{t >= s} dy[b, t, d] C[b, t, n]
    prod = dy.astype(np.float64)[..., None] * Cd[:, :, None, :]
    rev = np.flip(np.cumsum(np.flip(prod, axis=1), axis=1), axis=1)
    du = a["D"][None, None, :] * dy + dlt * np.einsum("bsn,bsdn->bsd", a["B"].astype(np.float64), rev)
    np.testing.assert_allclose(grads["du"], du, rtol=1e-12, atol=1e-13)
    dB = np.einsum("bsd,bsdn->bsn", dlt * a["u"], rev)
    np.testing.assert_allclose(grads["dB"], dB, rtol=1e-12, atol=1e-13)
