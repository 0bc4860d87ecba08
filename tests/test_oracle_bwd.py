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


def test_bwd_matches_the_derivative_of_the_unrolled_sum(oracle_mod):
    """Without the gate, the forward is the double sum h_t = Σ_{s≤t} e^{A(S_t − S_s)} Δ_s B_s u_s
    (S_t = Σ_{r≤t} Δ_r), y_t = Σ_n C_t h_t + D u_t.  Differentiating J = Σ dy·y + Σ dlast·h_{L−1}
    term by term, with G_t = dy_t C_t (+ dlast at t = L−1) and E_ts = e^{A(S_t − S_s)}:
      ∂J/∂u_s = D dy_s + Σ_n Δ_s B_s Σ_{t≥s} G_t E_ts          ∂J/∂B_s = Σ_d Δ_s u_s Σ_{t≥s} G_t E_ts
      ∂J/∂C_t = Σ_d dy_t h_t                                    ∂J/∂A  = Σ_t G_t Σ_{s≤t} (S_t − S_s) E_ts Δ_s B_s u_s
      ∂J/∂Δ_r = Σ_n Σ_{t≥r} G_t (B_r u_r E_tr + A Σ_{s<r} E_ts Δ_s B_s u_s)
    then dA_log = A·∂J/∂A, ∂J/∂δ_r = σ(δ_r + bias)·∂J/∂Δ_r, dbias = Σ ∂J/∂δ, dD = Σ dy·u.
    An independent derivation of the oracle's adjoint recurrence, with real decays."""
    batch, L, Dm, N = 2, 11, 3, 4
    a, _, dy, dlast = _problem(5, batch=batch, L=L, Dm=Dm, N=N, gate=False)
    g = oracle_mod.ss_bwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], None, dy,
                          dlast=dlast)
    f = lambda k: a[k].astype(np.float64)
    u, dr, Bm, Cm, D, bias = f("u"), f("delta_raw"), f("B"), f("C"), f("D"), f("delta_bias")
    A = -np.exp(f("A_log"))
    dyy = dy.astype(np.float64)
    want = {k: np.zeros_like(v) for k, v in (("du", u), ("ddelta_raw", u), ("dB", Bm), ("dC", Cm))}
    dA = np.zeros((Dm, N))
    for b in range(batch):
        for d in range(Dm):
            x = dr[b, :, d] + bias[d]
            dlt = np.logaddexp(0.0, x)
            S = np.cumsum(dlt)
            dDel = np.zeros(L)
            for n in range(N):
                E = np.exp(A[d, n] * (S[:, None] - S[None, :]))          # E[t, s]
                G = dyy[b, :, d] * Cm[b, :, n]
                G[-1] += dlast[b, d, n]
                w = dlt * Bm[b, :, n] * u[b, :, d]                      # Δ_s B_s u_s
                h = np.array([np.sum(E[t, :t + 1] * w[:t + 1]) for t in range(L)])
                back = np.array([np.sum(G[s:] * E[s:, s]) for s in range(L)])   # Σ_{t≥s} G_t E_ts
                want["du"][b, :, d] += dlt * Bm[b, :, n] * back
                want["dB"][b, :, n] += dlt * u[b, :, d] * back
                want["dC"][b, :, n] += dyy[b, :, d] * h
                dA[d, n] += sum(G[t] * np.sum((S[t] - S[:t + 1]) * E[t, :t + 1] * w[:t + 1]) for t in range(L))
                for r in range(L):
                    inner = np.array([np.sum(E[t, :r] * w[:r]) for t in range(r, L)])
                    dDel[r] += np.sum(G[r:] * (Bm[b, r, n] * u[b, r, d] * E[r:, r] + A[d, n] * inner))
            want["du"][b, :, d] += D[d] * dyy[b, :, d]
            want["ddelta_raw"][b, :, d] = dDel / (1.0 + np.exp(-x))
    for k in ("du", "ddelta_raw", "dB", "dC"):
        np.testing.assert_allclose(g[k], want[k], rtol=1e-11, atol=1e-12 * np.max(np.abs(want[k])), err_msg=k)
    np.testing.assert_allclose(g["dA_log"], dA * A, rtol=1e-11, atol=1e-12 * np.max(np.abs(dA)))
    np.testing.assert_allclose(g["dD"], np.sum(dyy * u, axis=(0, 1)), rtol=1e-12)
    np.testing.assert_allclose(g["ddelta_bias"], want["ddelta_raw"].sum(axis=(0, 1)), rtol=1e-11,
                               atol=1e-12 * np.max(np.abs(want["ddelta_raw"])))
