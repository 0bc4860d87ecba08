"""Parity of the CUDA backward scan (ss_bwd, through the C ABI) with the fp64 oracle's
gradients.  Elementwise gradients (du, ddelta_raw, dz, dh0) and the sums over channels or
batch rows (dB, dC, dA_log, dD, ddelta_bias, accumulated with atomics) have separate gates."""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import BF16_REL_L2, assert_fwd_close, f32dev, rel_l2, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GRAD_REL_L2 = 1e-5       # fp32, elementwise gradients
SUM_REL_L2 = 1e-4        # fp32 sums over channels / batch rows (atomic order varies)
BF16_SUM_REL_L2 = 1e-3

ELEMENTWISE = ("du", "ddelta_raw", "dz", "dh0")
SUMS = ("dB", "dC", "dA_log", "dD", "ddelta_bias")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def problem(batch, L, Dm, N, io="f32", seed=0, gate=True, with_h0=True, with_dlast=True, **kw):
    w = synth.fwd_inputs(batch, L, Dm, N, io=io, seed=seed, **kw)
    a = w.arrays
    if not gate:
        a["z"] = None
    g = synth.rng_for(seed, 12)
    dy = g.standard_normal((batch, L, Dm), dtype=np.float32)
    if io == "bf16":
        dy = synth.round_bf16(dy)
    h0 = synth.initial_state(batch, Dm, N, seed=seed) if with_h0 else None
    dlast = g.standard_normal((batch, Dm, N), dtype=np.float32) if with_dlast else None
    return w, a, dy, h0, dlast


def run(w, a, dy, h0, dlast):
    io = w.io
    t = dict(u=to_dev(a["u"], io), delta_raw=to_dev(a["delta_raw"], io), z=to_dev(a["z"], io),
             B=to_dev(a["B"], io), C=to_dev(a["C"], io))
    g = ss.ss_bwd(to_dev(dy, io), t["u"], t["delta_raw"], f32dev(a["delta_bias"]), f32dev(a["A_log"]), t["B"],
                  t["C"], f32dev(a["D"]), t["z"], h0=f32dev(h0), dlast=f32dev(dlast))
    torch.cuda.synchronize()
    return {k: (None if v is None else to_host(v)) for k, v in g.items()}


def reference(a, dy, h0, dlast):
    return oracle.ss_bwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"], dy,
                         h0=None if h0 is None else h0.astype(np.float64),
                         dlast=None if dlast is None else dlast.astype(np.float64))


def check(w, a, dy, h0, dlast, what=""):
    got = run(w, a, dy, h0, dlast)
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE + SUMS:
        if k == "dz" and a["z"] is None:
            assert got["dz"] is None
            continue
        if k == "dD" and a["D"] is None:
            continue
        assert np.all(np.isfinite(got[k])), f"{what} {k}: non-finite"
        e = rel_l2(got[k], ref[k])
        if w.io == "bf16":
            tol = BF16_REL_L2 if k in ("du", "ddelta_raw", "dz") else BF16_SUM_REL_L2
        else:
            tol = GRAD_REL_L2 if k in ELEMENTWISE else SUM_REL_L2
        assert e <= tol, f"{what} {k}: rel-L2 {e:.3e} > {tol}"
    return got, ref


class staging:
    """Pin how ss_bwd stages its tiles: -1 automatic, 0 plain loads, 1 TMA."""

    def __init__(self, v):
        self.v = v

    def __enter__(self):
        lib = ss.lib()
        lib.ss__force_bwd_tma.argtypes = [ctypes.c_int]
        self.prev = lib.ss__force_bwd_tma(self.v)

    def __exit__(self, *a):
        ss.lib().ss__force_bwd_tma(self.prev)


STAGINGS = pytest.mark.parametrize("stage", [-1, 0], ids=["auto", "plain"])


class splitting:
    """Pin the backward's time split: -1 automatic, 0 never, n >= 2 up to n segments."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        lib = ss.lib()
        lib.ss__force_bwd_nseg.argtypes = [ctypes.c_int]
        self.prev = lib.ss__force_bwd_nseg(self.n)

    def __exit__(self, *a):
        ss.lib().ss__force_bwd_nseg(self.prev)


SPLITS = pytest.mark.parametrize("nseg", [0, 3, -1], ids=["one-pass", "split3", "auto"])


@SPLITS
@STAGINGS
@pytest.mark.parametrize("L", [1, 5, 31, 32, 33, 63, 64, 65, 200])
def test_bwd_lengths(L, stage, nseg):
    with staging(stage), splitting(nseg):
        check(*problem(2, L, 40, 16, seed=L), what=f"L={L}")


@STAGINGS
@pytest.mark.parametrize("N", [1, 3, 4, 5, 8, 12, 16])
def test_bwd_state_counts(N, stage):
    with staging(stage):
        check(*problem(2, 130, 72, N, seed=20 + N), what=f"N={N}")


@STAGINGS
@pytest.mark.parametrize("Dm", [1, 31, 33, 100])
def test_bwd_channel_counts(Dm, stage):
    with staging(stage):
        check(*problem(3, 97, Dm, 16, seed=40 + Dm), what=f"Dm={Dm}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_tma_staging_taken(io):
    """Contiguous inputs with 16-byte rows are staged by TMA (forcing it is accepted), and
    both stagings give the same gradients up to the atomics' summation order."""
    w, a, dy, h0, dlast = problem(2, 200, 64, 16, io=io, seed=70)
    with staging(1):
        g1 = run(w, a, dy, h0, dlast)
    with staging(0):
        g0 = run(w, a, dy, h0, dlast)
    for k in ("du", "ddelta_raw", "dz", "dh0"):
        np.testing.assert_array_equal(g1[k], g0[k], err_msg=k)
    for k in SUMS:
        assert rel_l2(g1[k], g0[k]) <= 1e-6, k


def test_bwd_strided_inputs_fall_back_to_plain_staging():
    """u, δ, z as views with a row pitch of Dm + 1 floats (not a multiple of 16 bytes): TMA is
    refused when forced, and the automatic choice stages them with plain loads."""
    w, a, dy, h0, dlast = problem(2, 150, 48, 16, seed=71)
    wide = {k: np.zeros((2, 150, 49), np.float32) for k in ("u", "delta_raw", "z")}
    t = {}
    for k in wide:
        wide[k][..., :48] = a[k]
        t[k] = torch.from_numpy(wide[k]).cuda()[..., :48]
    args = (f32dev(dy), t["u"], t["delta_raw"], f32dev(a["delta_bias"]), f32dev(a["A_log"]), f32dev(a["B"]),
            f32dev(a["C"]), f32dev(a["D"]), t["z"])
    with staging(1):
        with pytest.raises(ss.SelscanError):
            ss.ss_bwd(*args, h0=f32dev(h0), dlast=f32dev(dlast))
    g = ss.ss_bwd(*args, h0=f32dev(h0), dlast=f32dev(dlast))
    torch.cuda.synchronize()
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE + SUMS:
        e = rel_l2(to_host(g[k]), ref[k])
        assert e <= (GRAD_REL_L2 if k in ELEMENTWISE else SUM_REL_L2), (k, e)


@SPLITS
@pytest.mark.parametrize("opts", ["no_gate", "no_h0", "no_dlast", "plain"])
def test_bwd_optional_inputs(opts, nseg):
    kw = dict(gate=opts not in ("no_gate", "plain"), with_h0=opts not in ("no_h0", "plain"),
              with_dlast=opts not in ("no_dlast", "plain"))
    with splitting(nseg):
        check(*problem(2, 150, 48, 16, seed=50, **kw), what=opts)


@pytest.mark.parametrize("nseg", [2, 5, 8, 64])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_time_split_segment_counts(nseg, io):
    """Forced segment counts (up to one per 32-step chunk) on a few-tile problem with h0 and
    dlast, against the oracle and against the one-pass schedule."""
    args = problem(1, 1000, 64, 16, io=io, seed=200 + nseg)
    with splitting(nseg):
        got, _ = check(*args, what=f"split {nseg} {io}")
    with splitting(0):
        one = run(*args)
    tol = 1e-5 if io == "f32" else 5e-3
    for k in ("du", "ddelta_raw", "dz", "dh0"):
        assert rel_l2(got[k], one[k]) <= tol, k


@STAGINGS
@pytest.mark.parametrize("N", [4, 16])
def test_bwd_bf16(N, stage):
    with staging(stage):
        check(*problem(2, 300, 64, N, io="bf16", seed=60 + N), what="bf16")


@pytest.mark.parametrize("nseg", [0, -1], ids=["one-pass", "auto"])
def test_bwd_long_sequence(nseg):
    with splitting(nseg):
        check(*problem(2, 2048, 256, 16, seed=61), what="L=2048")


def test_bwd_long32k_shape_sampled():
    """The long-sequence shape (batch 1, L 32768, Dm 1536, N 16) on the automatic time split:
    dh0 and dA_log against the oracle on a channel slice (the oracle runs the sliced problem,
    which the slice's gradients depend on alone), the elementwise gradients on that slice too."""
    w = synth.config("long32k")
    a = w.arrays
    dy = synth.rng_for(63, 12).standard_normal((1, w.L, w.Dm), dtype=np.float32)
    got = run(w, a, dy, None, None)
    sl = slice(0, 64)
    sub = {k: (None if v is None else (v[..., sl] if v.ndim == 3 and v.shape[-1] == w.Dm else
                                       v[sl] if v.shape[0] == w.Dm else v)) for k, v in a.items()}
    ref = oracle.ss_bwd(sub["u"], sub["delta_raw"], sub["delta_bias"], sub["A_log"], sub["B"], sub["C"], sub["D"],
                        sub["z"], dy[..., sl])
    for k in ("du", "ddelta_raw", "dz"):
        assert rel_l2(got[k][..., sl], ref[k]) <= GRAD_REL_L2, k
    for k in ("dA_log", "dD", "ddelta_bias"):
        assert rel_l2(got[k][sl], ref[k]) <= SUM_REL_L2, k


def test_bwd_full_size_130m():
    """The 130m-shaped layer (batch 8, L 2048, Dm 1536, N 16), gradients of every input."""
    w = synth.config("mamba130m")
    g = synth.rng_for(62, 12)
    dy = g.standard_normal((w.batch, w.L, w.Dm), dtype=np.float32)
    check(w, w.arrays, dy, None, None, what="130m")


def test_bwd_matches_forward_difference_on_gpu():
    """The GPU gradient of sum(dy * y) in a random direction v of u matches the directional
    difference of two GPU forward passes (step 1e-3, central), a check that does not go
    through the oracle."""
    w, a, dy, _, _ = problem(2, 300, 64, 16, seed=63, with_h0=False, with_dlast=False)
    got = run(w, a, dy, None, None)
    v = synth.rng_for(64, 12).standard_normal(a["u"].shape).astype(np.float32)
    eps = 1e-3

    def J(u):
        t = {k: f32dev(a[k]) for k in ("delta_raw", "z", "B", "C", "A_log", "D", "delta_bias")}
        y = ss.ss_fwd(f32dev(u), t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"])
        torch.cuda.synchronize()
        return float(np.sum(to_host(y) * dy.astype(np.float64)))
    fd = (J(a["u"] + eps * v) - J(a["u"] - eps * v)) / (2 * eps)
    an = float(np.sum(got["du"] * v))
    assert abs(fd - an) <= 1e-3 * abs(an) + 1e-3, (fd, an)


def test_bwd_rejects_small_workspace_and_overlap():
    w, a, dy, h0, dlast = problem(1, 64, 32, 16, seed=65)
    lib = ss.lib()
    t = {k: f32dev(v) for k, v in a.items() if v is not None}
    dyd = f32dev(dy)
    out = {k: torch.empty(sh, device="cuda") for k, sh in (("du", (1, 64, 32)), ("dd", (1, 64, 32)), ("dz", (1, 64, 32)),
                                                          ("dB", (1, 64, 16)), ("dC", (1, 64, 16)), ("dA", (32, 16)))}
    s = ss.FwdStrides(ss.SS_F32, 64 * 32, 32, 64 * 32, 32, 64 * 32, 32, 0, 0, 64 * 16, 16, 64 * 16, 16)
    need = lib.ss_bwd_workspace_size(1, 64, 32, 16)
    ws = torch.zeros(need + 256, dtype=torch.uint8, device="cuda")

    def call(du_ptr, nbytes):
        return lib.ss_bwd(t["u"].data_ptr(), t["delta_raw"].data_ptr(), t["delta_bias"].data_ptr(),
                          t["A_log"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(), t["D"].data_ptr(),
                          t["z"].data_ptr(), None, dyd.data_ptr(), None, du_ptr, out["dd"].data_ptr(),
                          out["dz"].data_ptr(), out["dB"].data_ptr(), out["dC"].data_ptr(), out["dA"].data_ptr(),
                          None, None, None, 1, 64, 32, 16, ctypes.byref(s), ws.data_ptr(), nbytes, None)
    assert call(out["du"].data_ptr(), need - 4) == 1          # workspace too small
    assert call(t["u"].data_ptr(), need) == 1                 # du over an input
    assert call(out["dd"].data_ptr(), need) == 1              # du over ddelta_raw
    assert call(out["du"].data_ptr(), need) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("N", [16, 6])
def test_bwd_sums_at_4_byte_offsets(N):
    """dB and dC 4-byte but not 16-byte aligned (and N not a multiple of 4): the kernel's scalar
    atomics instead of its 16-byte reductions give the same sums."""
    batch, L, Dm = 2, 80, 40
    w, a, dy, h0, dlast = problem(batch, L, Dm, N, seed=66, with_h0=False, with_dlast=False)
    lib = ss.lib()
    t = {k: f32dev(v) for k, v in a.items() if v is not None}
    dyd = f32dev(dy)
    x = (batch, L, Dm)
    du, dd, dz = (torch.empty(x, device="cuda") for _ in range(3))
    dA = torch.empty((Dm, N), device="cuda")
    n = batch * L * N
    bc = torch.full((2 * n + 8,), float("nan"), device="cuda")
    dB, dC = bc[1:1 + n], bc[n + 5:2 * n + 5]             # element offsets 1 and n + 5: never 16-byte aligned
    s = ss.FwdStrides(ss.SS_F32, L * Dm, Dm, L * Dm, Dm, L * Dm, Dm, 0, 0, L * N, N, L * N, N)
    need = lib.ss_bwd_workspace_size(batch, L, Dm, N)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = lib.ss_bwd(t["u"].data_ptr(), t["delta_raw"].data_ptr(), t["delta_bias"].data_ptr(), t["A_log"].data_ptr(),
                    t["B"].data_ptr(), t["C"].data_ptr(), t["D"].data_ptr(), t["z"].data_ptr(), None, dyd.data_ptr(),
                    None, du.data_ptr(), dd.data_ptr(), dz.data_ptr(), dB.data_ptr(), dC.data_ptr(), dA.data_ptr(),
                    None, None, None, batch, L, Dm, N, ctypes.byref(s), ws.data_ptr(), need, None)
    assert st == 0
    torch.cuda.synchronize()
    ref = reference(a, dy, None, None)
    assert rel_l2(to_host(dB).reshape(batch, L, N), ref["dB"]) <= SUM_REL_L2
    assert rel_l2(to_host(dC).reshape(batch, L, N), ref["dC"]) <= SUM_REL_L2
    assert rel_l2(to_host(du), ref["du"]) <= GRAD_REL_L2
    assert torch.isnan(bc[0]) and torch.isnan(bc[n + 1:n + 5]).all() and torch.isnan(bc[2 * n + 5:]).all()


def run_with_ckpt(w, a, dy, h0, dlast, rows=None):
    """ss_fwd_ckpt (its y and last_state against the oracle's forward, on `rows` channels when
    given) then ss_bwd with its checkpoints."""
    io = w.io
    t = dict(u=to_dev(a["u"], io), delta_raw=to_dev(a["delta_raw"], io), z=to_dev(a["z"], io),
             B=to_dev(a["B"], io), C=to_dev(a["C"], io))
    prm = dict(delta_bias=f32dev(a["delta_bias"]), A_log=f32dev(a["A_log"]), D=f32dev(a["D"]))
    h0d = f32dev(h0)
    last = torch.empty((w.batch, w.Dm, w.N), device="cuda")
    y, ckpt = ss.ss_fwd_ckpt(t["u"], t["delta_raw"], prm["delta_bias"], prm["A_log"], t["B"], t["C"], prm["D"],
                             t["z"], last_state=last, h0=h0d)
    torch.cuda.synchronize()
    ry, rl, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"],
                                h0=None if h0 is None else h0.astype(np.float64), rows=rows)
    yh, lh = to_host(y), to_host(last)
    if rows is not None:
        yh, lh = yh[0][:, rows].T, lh[0][rows]
    assert_fwd_close(io, yh, ry, mag, lh, rl, what=f"ss_fwd_ckpt {w.name}")
    g = ss.ss_bwd(to_dev(dy, io), t["u"], t["delta_raw"], prm["delta_bias"], prm["A_log"], t["B"], t["C"], prm["D"],
                  t["z"], h0=h0d, dlast=f32dev(dlast), ckpt=ckpt)
    torch.cuda.synchronize()
    return {k: (None if v is None else to_host(v)) for k, v in g.items()}


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 15, 16, 33, 64, 65, 200, 1000])
def test_bwd_with_forward_checkpoints(io, L):
    """The backward from the forward's checkpoints (no first pass of its own) against the oracle,
    with h0 and dlast, on ragged lengths (entries past the last step hold the final state)."""
    w, a, dy, h0, dlast = problem(2, L, 200, 16, io=io, seed=70 + L)
    got = run_with_ckpt(w, a, dy, h0, dlast)
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE + SUMS:
        e = rel_l2(got[k], ref[k])
        if io == "bf16":
            tol = BF16_REL_L2 if k in ("du", "ddelta_raw", "dz") else BF16_SUM_REL_L2
        else:
            tol = GRAD_REL_L2 if k in ELEMENTWISE else SUM_REL_L2
        assert e <= tol, f"ckpt L={L} {io} {k}: rel-L2 {e:.3e} > {tol}"


def test_bwd_with_forward_checkpoints_130m_equals_plain_backward():
    """The 130m-shaped layer: with the forward's checkpoints the elementwise gradients equal the
    backward's own (its first pass folds the same steps with the same arithmetic), the sums up to
    their atomic order; and the oracle's on sampled channels."""
    w = synth.config("mamba130m")
    a = w.arrays
    dy = synth.rng_for(71, 12).standard_normal((w.batch, w.L, w.Dm), dtype=np.float32)
    got = run_with_ckpt(w, a, dy, None, None, rows=np.sort(np.random.default_rng(7).choice(w.Dm, 16, replace=False)))
    plain = run(w, a, dy, None, None)
    for k in ELEMENTWISE:
        if got[k] is not None:
            assert rel_l2(got[k], plain[k]) <= 1e-6, k
    for k in SUMS:
        assert rel_l2(got[k], plain[k]) <= 1e-5, k


def test_fwd_ckpt_refusals_and_split_backward():
    """N other than 16 is refused by both calls; a backward that takes the time split (one long
    row) takes its segments' entering states from the checkpoints (the local launch sweeps only
    the adjoint, summing Δ as it goes) and gives the oracle's gradients."""
    w5, a5, dy5, _, _ = problem(1, 40, 32, 8, seed=72, with_h0=False, with_dlast=False)
    assert ss.lib().ss_fwd_ckpt_size(1, 40, 32, 8) == 0
    with pytest.raises(ss.SelscanError):
        ss.ss_fwd_ckpt(f32dev(a5["u"]), f32dev(a5["delta_raw"]), f32dev(a5["delta_bias"]), f32dev(a5["A_log"]),
                       f32dev(a5["B"]), f32dev(a5["C"]), f32dev(a5["D"]), f32dev(a5["z"]),
                       ckpt=torch.empty(1024, device="cuda"))
    w, a, dy, h0, dlast = problem(1, 3000, 64, 16, seed=73)
    with splitting(4):
        got = run_with_ckpt(w, a, dy, h0, dlast)
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE:
        assert rel_l2(got[k], ref[k]) <= GRAD_REL_L2, k
    for k in SUMS:
        assert rel_l2(got[k], ref[k]) <= SUM_REL_L2, k


@pytest.mark.parametrize("nseg", [2, 5])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_split_with_forward_checkpoints(nseg, io):
    """The time split from the forward's checkpoints at forced segment counts, ragged length,
    with h0 and dlast, against the oracle."""
    w, a, dy, h0, dlast = problem(2, 1500, 96, 16, io=io, seed=74 + nseg)
    with splitting(nseg):
        got = run_with_ckpt(w, a, dy, h0, dlast)
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE + SUMS:
        e = rel_l2(got[k], ref[k])
        if io == "bf16":
            tol = BF16_REL_L2 if k in ("du", "ddelta_raw", "dz") else BF16_SUM_REL_L2
        else:
            tol = GRAD_REL_L2 if k in ELEMENTWISE else SUM_REL_L2
        assert e <= tol, f"split {nseg} {io} {k}: rel-L2 {e:.3e} > {tol}"


@pytest.mark.parametrize("io,batch", [("f32", 2), ("bf16", 4)])
def test_bwd_ckpt_balanced_forward(io, batch):
    """Enough tiles for ss_fwd_ckpt to take the balanced schedule with its workspace (fp32 on
    32-channel tiles at 4 lanes, bf16 with fp32 B/C tiles at 2): y bit for bit ss_fwd's on the
    same schedule, and the backward from its checkpoints against the oracle."""
    w, a, dy, h0, dlast = problem(batch, 100, 4864, 16, io=io, seed=80 + batch)
    t = dict(u=to_dev(a["u"], io), delta_raw=to_dev(a["delta_raw"], io), z=to_dev(a["z"], io),
             B=to_dev(a["B"], io), C=to_dev(a["C"], io))
    prm = dict(delta_bias=f32dev(a["delta_bias"]), A_log=f32dev(a["A_log"]), D=f32dev(a["D"]))
    h0d = f32dev(h0)
    y1 = ss.ss_fwd(t["u"], t["delta_raw"], prm["delta_bias"], prm["A_log"], t["B"], t["C"], prm["D"], t["z"],
                   h0=h0d, workspace=True)
    y2, ckpt = ss.ss_fwd_ckpt(t["u"], t["delta_raw"], prm["delta_bias"], prm["A_log"], t["B"], t["C"], prm["D"],
                              t["z"], h0=h0d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(y1), to_host(y2))
    g = ss.ss_bwd(to_dev(dy, io), t["u"], t["delta_raw"], prm["delta_bias"], prm["A_log"], t["B"], t["C"], prm["D"],
                  t["z"], h0=h0d, dlast=f32dev(dlast), ckpt=ckpt)
    torch.cuda.synchronize()
    got = {k: (None if v is None else to_host(v)) for k, v in g.items()}
    ref = reference(a, dy, h0, dlast)
    for k in ELEMENTWISE + SUMS:
        e = rel_l2(got[k], ref[k])
        if io == "bf16":
            tol = BF16_REL_L2 if k in ("du", "ddelta_raw", "dz") else BF16_SUM_REL_L2
        else:
            tol = GRAD_REL_L2 if k in ELEMENTWISE else SUM_REL_L2
        assert e <= tol, f"balanced ckpt {io} {k}: rel-L2 {e:.3e} > {tol}"


def test_fwd_ckpt_argument_checks():
    """ss_fwd_ckpt refuses time-invariant B/C and strides TMA cannot describe (no substitute
    schedule), a missing or misaligned checkpoint buffer, and one that overlaps y."""
    w, a, dy, h0, dlast = problem(2, 64, 64, 16, seed=90, with_h0=False, with_dlast=False)
    t = {k: f32dev(v) for k, v in a.items() if v is not None}
    need = ss.lib().ss_fwd_ckpt_size(2, 64, 64, 16)
    assert need == 2 * 2 * 2 * 2 * 32 * 16 * 4
    ck = torch.empty(need // 4 + 8, device="cuda")
    call = lambda **kw: ss.ss_fwd_ckpt(kw.get("u", t["u"]), t["delta_raw"], t["delta_bias"], t["A_log"],
                                       kw.get("B", t["B"]), kw.get("C", t["C"]), t["D"], t["z"], y=kw.get("y"),
                                       ckpt=kw.get("ckpt", ck[: need // 4]), workspace=False)
    call()
    torch.cuda.synchronize()
    with pytest.raises(ss.SelscanError):                      # B, C at step stride 0
        call(B=t["B"][:, :1].expand(-1, 64, -1), C=t["C"][:, :1].expand(-1, 64, -1))
    wide = torch.zeros((2, 64, 66), device="cuda")
    wide[..., :64] = t["u"]
    with pytest.raises(ss.SelscanError):                      # rows 264 bytes apart: no TMA
        call(u=wide[..., :64])
    with pytest.raises(ss.SelscanError):                      # 4 bytes off 16-byte alignment
        call(ckpt=ck[1: 1 + need // 4])
    yb = torch.empty(need // 4 + 2 * 64 * 64, device="cuda")
    with pytest.raises(ss.SelscanError):                      # y over the checkpoints
        call(y=yb[: 2 * 64 * 64].view(2, 64, 64), ckpt=yb[: need // 4])
    lib = ss.lib()
    s = ss.FwdStrides(ss.SS_F32, 64 * 64, 64, 64 * 64, 64, 64 * 64, 64, 64 * 64, 64, 64 * 16, 16, 64 * 16, 16)
    y = torch.empty((2, 64, 64), device="cuda")
    assert lib.ss_fwd_ckpt(t["u"].data_ptr(), t["delta_raw"].data_ptr(), None, t["A_log"].data_ptr(),
                           t["B"].data_ptr(), t["C"].data_ptr(), None, None, y.data_ptr(), None, None, None,
                           2, 64, 64, 16, ctypes.byref(s), None, 0, None) == 1    # no checkpoint buffer
