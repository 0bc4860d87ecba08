"""Time-invariant B and C (step stride 0: the linear time-invariant case that the official
kernel specialises with its kIsVariableB/C branch): the forward scan against the oracle on the
same values written out per step, the register-held B/C kernel against the generic fill, the
forward against the convolution form of an LTI system, and the backward scan."""
import ctypes

import numpy as np
import pytest
from scipy.special import expit

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import assert_fwd_close, f32dev, rel_l2, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


class ForceVariant:
    def __init__(self, family=-1, lpc=0, tma=-1):
        self.args = (family, lpc, tma)

    def __enter__(self):
        f = ss.lib().ss__force_fwd_variant
        f.argtypes = [ctypes.c_int] * 3
        assert f(*self.args) == 0

    def __exit__(self, *exc):
        ss.lib().ss__force_fwd_variant(-1, 0, -1)


def lti_problem(batch, L, Dm, N, io="f32", seed=0, lti_c=True):
    """Seeded inputs whose B (and C) rows are the same at every step of a batch row; the
    arrays hold those values written out per step (what the oracle reads)."""
    w = synth.fwd_inputs(batch, L, Dm, N, io=io, seed=seed)
    a = w.arrays
    a["B"] = np.broadcast_to(a["B"][:, :1], (batch, L, N)).copy()
    if lti_c:
        a["C"] = np.broadcast_to(a["C"][:, :1], (batch, L, N)).copy()
    return w, a


def stride0(arr, io):
    """[batch, L, N] with equal rows -> a [batch, L, N] view of one row per batch (step stride 0)."""
    return to_dev(arr[:, :1], io).expand(-1, arr.shape[1], -1)


def run(w, a, variant=(-1, 0, -1), workspace=False, lti_c=True):
    io = w.io
    Bm = stride0(a["B"], io)
    Cm = stride0(a["C"], io) if lti_c else to_dev(a["C"], io)
    assert Bm.stride(1) == 0 or w.L == 1
    last = torch.full((w.batch, w.Dm, w.N), float("nan"), device="cuda")
    with ForceVariant(*variant):
        y = ss.ss_fwd(to_dev(a["u"], io), to_dev(a["delta_raw"], io), f32dev(a["delta_bias"]), f32dev(a["A_log"]),
                      Bm, Cm, f32dev(a["D"]), to_dev(a["z"], io), last_state=last, workspace=workspace)
    torch.cuda.synchronize()
    return to_host(y), to_host(last)


def check_oracle(w, a, y, last, what):
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"])
    assert_fwd_close(w.io, y, ry, mag, last, rl, what=what)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("lpc", [1, 2, 4])
def test_lti_kernel_against_oracle_and_generic_fill(io, lpc):
    w, a = lti_problem(2, 300, 100, 16, io=io, seed=80 + lpc)
    y, last = run(w, a, variant=(0, lpc, -1))
    check_oracle(w, a, y, last, f"lti {io} lpc={lpc}")
    y0, last0 = run(w, a, variant=(0, lpc, 0))        # plain-load fill reading B/C at stride 0
    np.testing.assert_array_equal(y, y0)
    np.testing.assert_array_equal(last, last0)


@pytest.mark.parametrize("N", [1, 4, 5, 8, 12])
def test_lti_state_counts(N):
    w, a = lti_problem(2, 130, 72, N, seed=90 + N)
    y, last = run(w, a)
    check_oracle(w, a, y, last, f"lti N={N}")


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 2049])
def test_lti_lengths(L):
    w, a = lti_problem(2, L, 40, 16, seed=100 + L)
    y, last = run(w, a)
    check_oracle(w, a, y, last, f"lti L={L}")


def test_lti_with_workspace_is_the_per_tile_schedule():
    w, a = lti_problem(4, 500, 256, 16, seed=110)
    y, last = run(w, a)
    yw, lw = run(w, a, workspace=True)
    np.testing.assert_array_equal(y, yw)
    np.testing.assert_array_equal(last, lw)


def test_lti_few_rows_long_sequence():
    """One row, a long sequence: the segment family (generic fill) or, with a workspace, no
    time split (the LTI kernel runs per tile)."""
    w, a = lti_problem(1, 4000, 64, 16, seed=111)
    y, last = run(w, a)
    check_oracle(w, a, y, last, "lti seg")
    yw, lw = run(w, a, workspace=True)
    check_oracle(w, a, yw, lw, "lti seg ws")


def test_only_B_time_invariant():
    w, a = lti_problem(2, 200, 64, 16, seed=112, lti_c=False)
    y, last = run(w, a, lti_c=False)
    check_oracle(w, a, y, last, "B only")


def test_lti_forward_is_a_causal_convolution():
    """Not through the oracle: with Δ constant over the steps too, y = silu(z)·(K * u) with
    K_k = Σ_n C_n a_n^k Δ B_n (+ D at k = 0), computed with numpy.convolve in fp64."""
    batch, L, Dm, N = 2, 200, 8, 16
    w, a = lti_problem(batch, L, Dm, N, seed=113)
    g = np.random.default_rng(7)
    a["delta_raw"] = np.broadcast_to(g.standard_normal((1, 1, Dm)).astype(np.float32), (batch, L, Dm)).copy()
    y, _ = run(w, a)
    ref = np.zeros((batch, L, Dm))
    for b in range(batch):
        for d in range(Dm):
            dlt = np.logaddexp(0.0, float(a["delta_raw"][0, 0, d]) + float(a["delta_bias"][d]))
            A = -np.exp(a["A_log"][d].astype(np.float64))
            K = (a["C"][b, 0].astype(np.float64) * dlt * a["B"][b, 0].astype(np.float64)
                 * np.exp(dlt * A) ** np.arange(L)[:, None]).sum(axis=1)
            K[0] += float(a["D"][d])
            z = a["z"][b, :, d].astype(np.float64)
            ref[b, :, d] = np.convolve(a["u"][b, :, d].astype(np.float64), K)[:L] * z * expit(z)
    assert rel_l2(y, ref) <= 1e-5


def test_lti_backward():
    """ss_bwd with B, C at step stride 0: every gradient against the oracle (dB, dC per step;
    the gradient of the time-invariant row is their sum over the steps)."""
    w, a = lti_problem(2, 200, 64, 16, seed=114)
    dy = synth.rng_for(114, 12).standard_normal((w.batch, w.L, w.Dm), dtype=np.float32)
    g = ss.ss_bwd(f32dev(dy), f32dev(a["u"]), f32dev(a["delta_raw"]), f32dev(a["delta_bias"]), f32dev(a["A_log"]),
                  stride0(a["B"], "f32"), stride0(a["C"], "f32"), f32dev(a["D"]), f32dev(a["z"]))
    torch.cuda.synchronize()
    ref = oracle.ss_bwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"], dy)
    for k, tol in (("du", 1e-5), ("ddelta_raw", 1e-5), ("dz", 1e-5), ("dB", 1e-4), ("dC", 1e-4), ("dA_log", 1e-4),
                   ("dD", 1e-4), ("ddelta_bias", 1e-4)):
        e = rel_l2(to_host(g[k]), ref[k])
        assert e <= tol, (k, e)
    # the time-invariant row's gradient
    assert rel_l2(to_host(g["dB"]).sum(axis=1), ref["dB"].sum(axis=1)) <= 1e-4
