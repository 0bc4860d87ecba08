"""Parity of the forward scan with the low-rank time-step projection folded in
(ss_fwd_dtproj: delta_raw = dt_low · W_dt^T computed inside the kernel) with the fp64 oracle
that sums the projection in fp64."""
import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import assert_fwd_close, f32dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


def dtproj_problem(batch, L, Dm, N, R, seed):
    """Seeded inputs; dt_low ~ N(0, 0.5²) and W_dt ~ N(0, 1/R), so the projected time step has
    the spread of the plain workloads' delta_raw."""
    w = synth.fwd_inputs(batch, L, Dm, N, seed=seed)
    g = synth.rng_for(seed, 13)
    dt_low = (0.5 * g.standard_normal((batch, L, R))).astype(np.float32)
    W = (g.standard_normal((Dm, R)) / np.sqrt(R)).astype(np.float32)
    return w, w.arrays, dt_low, W


def run(w, a, dt_low, W, h0=None):
    last = torch.full((w.batch, w.Dm, w.N), float("nan"), device="cuda")
    y = ss.ss_fwd_dtproj(f32dev(a["u"]), f32dev(dt_low), f32dev(W), f32dev(a["delta_bias"]), f32dev(a["A_log"]),
                         f32dev(a["B"]), f32dev(a["C"]), f32dev(a["D"]), f32dev(a["z"]), last_state=last,
                         h0=f32dev(h0))
    torch.cuda.synchronize()
    return to_host(y), to_host(last)


def check(w, a, dt_low, W, what, h0=None):
    y, last = run(w, a, dt_low, W, h0=h0)
    ry, rl, mag = oracle.ss_fwd_dtproj(a["u"], dt_low, W, a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                       a["z"], h0=None if h0 is None else h0.astype(np.float64))
    assert_fwd_close("f32", y, ry, mag, last, rl, what=what)


@pytest.mark.parametrize("R", [4, 8, 12, 16, 48, 64])
def test_dtproj_ranks(R):
    check(*dtproj_problem(2, 300, 100, 16, R, seed=120 + R), what=f"R={R}")


@pytest.mark.parametrize("N", [1, 4, 5, 8, 12])
def test_dtproj_state_counts(N):
    # N not 4, 8, 16 cannot use TMA-fed B/C tiles: refused
    w, a, dt_low, W = dtproj_problem(2, 130, 72, N, 16, seed=130 + N)
    if N in (4, 8):
        check(w, a, dt_low, W, what=f"N={N}")
    else:
        with pytest.raises(ss.SelscanError):
            run(w, a, dt_low, W)


@pytest.mark.parametrize("L", [1, 47, 48, 49, 97, 2049])
def test_dtproj_lengths(L):
    check(*dtproj_problem(2, L, 40, 16, 16, seed=140 + L), what=f"L={L}")


@pytest.mark.parametrize("Dm", [4, 36, 100, 200])
def test_dtproj_channel_counts(Dm):
    """Channel counts that leave a partial last tile (rows must be whole 16-byte units for TMA)."""
    check(*dtproj_problem(3, 97, Dm, 16, 48, seed=150 + Dm), what=f"Dm={Dm}")


def test_dtproj_few_rows_and_h0():
    """One row (the lane kernel at 4 lanes per channel regardless) from an initial state."""
    w, a, dt_low, W = dtproj_problem(1, 1000, 64, 16, 48, seed=160)
    h0 = synth.initial_state(1, 64, 16, seed=160)
    check(w, a, dt_low, W, what="h0", h0=h0)


def test_dtproj_equals_plain_forward_on_an_exact_projection():
    """Not through the oracle: dt_low and W on a 2^-4 grid make the fp32 projection exact, so
    ss_fwd fed that projection and ss_fwd_dtproj see the same time steps; they agree to the
    fp32 accuracy of one scan."""
    w, a, _, _ = dtproj_problem(2, 500, 96, 16, 8, seed=161)
    g = np.random.default_rng(161)
    dt_low = (g.integers(-32, 33, size=(2, 500, 8)) / 16).astype(np.float32)
    W = (g.integers(-32, 33, size=(96, 8)) / 16).astype(np.float32) / 4
    dr = (dt_low.astype(np.float64) @ W.T.astype(np.float64)).astype(np.float32)
    y1, l1 = run(w, a, dt_low, W)
    y0 = to_host(ss.ss_fwd(f32dev(a["u"]), f32dev(dr), f32dev(a["delta_bias"]), f32dev(a["A_log"]), f32dev(a["B"]),
                           f32dev(a["C"]), f32dev(a["D"]), f32dev(a["z"])))
    torch.cuda.synchronize()
    np.testing.assert_allclose(y1, y0, rtol=2e-5, atol=2e-5 * np.abs(y0).max())


def test_dtproj_rejects_unsupported():
    w, a, dt_low, W = dtproj_problem(1, 64, 32, 16, 16, seed=162)
    with pytest.raises(ss.SelscanError):          # rank not a multiple of 4
        run(w, a, dt_low[..., :6].copy(), W[:, :6].copy())
    with pytest.raises(ss.SelscanError):          # rank above 64
        run(w, a, np.zeros((1, 64, 68), np.float32), np.zeros((32, 68), np.float32))
    w2, a2, d2, W2 = dtproj_problem(1, 64, 33, 16, 16, seed=163)
    with pytest.raises(ss.SelscanError):          # 33-channel rows: not whole 16-byte units
        run(w2, a2, d2, W2)
    with pytest.raises(ss.SelscanError):          # bf16 I/O
        ss.ss_fwd_dtproj(f32dev(a["u"]).bfloat16(), f32dev(dt_low), f32dev(W), None, f32dev(a["A_log"]),
                         f32dev(a["B"]).bfloat16(), f32dev(a["C"]).bfloat16())
