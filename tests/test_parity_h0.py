"""Parity of the forward scan from an initial state (ss_fwd_h0) and of the time-split schedule
(ss_fwd_ws on shapes with few channel tiles) with the fp64 oracle, through the C ABI."""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import FP32_REL_L2, assert_fwd_close, f32dev, rel_l2, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


class Force:
    """Pin the forward kernel (family, lanes per channel, fill) and the time-split segment
    count (-1 automatic, 0 never, n >= 2 always)."""
    def __init__(self, family=-1, lpc=0, tma=-1, nseg=-1):
        self.v, self.nseg = (family, lpc, tma), nseg

    def __enter__(self):
        lib = ss.lib()
        lib.ss__force_fwd_variant.argtypes = [ctypes.c_int] * 3
        lib.ss__force_nseg.argtypes = [ctypes.c_int]
        assert lib.ss__force_fwd_variant(*self.v) == 0
        lib.ss__force_nseg(self.nseg)

    def __exit__(self, *exc):
        ss.lib().ss__force_fwd_variant(-1, 0, -1)
        ss.lib().ss__force_nseg(-1)


def dev(w):
    a = w.arrays
    return dict(u=to_dev(a["u"], w.io), delta_raw=to_dev(a["delta_raw"], w.io), z=to_dev(a["z"], w.io),
                B=to_dev(a["B"], w.io), C=to_dev(a["C"], w.io), A_log=f32dev(a["A_log"]),
                D=f32dev(a["D"]), delta_bias=f32dev(a["delta_bias"]))


def gpu(w, h0=None, workspace=True, force=Force(), t=None, in_place=False):
    t = t or dev(w)
    last = torch.full((w.batch, w.Dm, w.N), float("nan"), device="cuda")
    h0d = None
    if h0 is not None:
        h0d = torch.from_numpy(np.ascontiguousarray(h0, np.float32)).cuda()
        if in_place:
            last = h0d
    with force:
        y = ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                      last_state=last, workspace=workspace, h0=h0d)
    torch.cuda.synchronize()
    return to_host(y), to_host(last)


def ref(w, h0=None):
    a = w.arrays
    return oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"], a["z"],
                         h0=None if h0 is None else np.asarray(h0, np.float64))


def check(w, h0=None, **kw):
    y, last = gpu(w, h0, **kw)
    ry, rlast, mag = ref(w, h0)
    assert_fwd_close(w.io, y, ry, mag, last, rlast, what=f"{w.name} b={w.batch} L={w.L} Dm={w.Dm} "
                                                         f"N={w.N} {w.io} {kw}")
    return y, last


VARIANTS = [(0, 1, 1), (0, 2, 1), (0, 4, 1), (1, 0, 1), (0, 1, 0), (0, 2, 0), (0, 4, 0), (1, 0, 0)]
VARIANT_IDS = ["lane1-tma", "lane2-tma", "lane4-tma", "seg-tma", "lane1-plain", "lane2-plain",
               "lane4-plain", "seg-plain"]


# ------------------------------------------------------------------ initial state, every kernel

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_h0_every_kernel_variant(io, variant):
    w = synth.fwd_inputs(2, 531, 72, 16, io=io, seed=41)
    check(w, synth.initial_state(2, 72, 16, seed=41), workspace=False, force=Force(*variant, nseg=0))


@pytest.mark.parametrize("N", [3, 4, 8, 12])
def test_h0_small_state_counts(N):
    w = synth.fwd_inputs(2, 203, 40, N, seed=42 + N)
    h0 = synth.initial_state(2, 40, N, seed=42 + N)
    fill = 1 if N in (4, 8, 16) else -1            # TMA tiles need N == the kernel's state width
    for variant in [(0, 1, fill), (1, 0, fill), (0, 1, 0)]:
        check(w, h0, workspace=False, force=Force(*variant, nseg=0))


def test_h0_balanced_schedule():
    w = synth.fwd_inputs(6, 1000, 4096, 16, seed=43)       # ranges split tiles between CTAs
    check(w, synth.initial_state(6, 4096, 16, seed=43), workspace=True, force=Force(nseg=0))


def test_h0_zero_equals_no_h0():
    w = synth.fwd_inputs(2, 300, 96, 16, seed=44)
    y1, l1 = gpu(w, None, workspace=False)
    y2, l2 = gpu(w, np.zeros((2, 96, 16), np.float32), workspace=False)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("k", [64, 700, 1001])
@pytest.mark.parametrize("workspace", [False, True], ids=["per-tile", "workspace"])
def test_split_across_calls_equals_one_call(k, workspace):
    """Chunked prefill: steps [0, k) then [k, L) from the first call's last_state give the
    one-call result (up to rounding) and match the oracle."""
    w = synth.fwd_inputs(2, 1500, 128, 16, seed=45)
    t = dev(w)
    y_full, last_full = gpu(w, workspace=workspace, t=t)
    seq = ("u", "delta_raw", "z", "B", "C")
    t1 = {key: (v[:, :k].contiguous() if key in seq else v) for key, v in t.items()}
    t2 = {key: (v[:, k:].contiguous() if key in seq else v) for key, v in t.items()}
    last1 = torch.empty((2, 128, 16), device="cuda")
    y1 = ss.ss_fwd(t1["u"], t1["delta_raw"], t1["delta_bias"], t1["A_log"], t1["B"], t1["C"], t1["D"], t1["z"],
                   last_state=last1, workspace=workspace)
    last2 = torch.empty((2, 128, 16), device="cuda")
    y2 = ss.ss_fwd(t2["u"], t2["delta_raw"], t2["delta_bias"], t2["A_log"], t2["B"], t2["C"], t2["D"], t2["z"],
                   last_state=last2, workspace=workspace, h0=last1)
    torch.cuda.synchronize()
    y_split = np.concatenate([to_host(y1), to_host(y2)], axis=1)
    assert rel_l2(y_split, y_full) <= FP32_REL_L2
    assert rel_l2(to_host(last2), last_full) <= FP32_REL_L2
    ry, rlast, mag = ref(w)
    assert_fwd_close("f32", y_split, ry, mag, to_host(last2), rlast, what=f"split at {k}")


@pytest.mark.parametrize("schedule", ["lane", "seg", "balanced", "timesplit"])
def test_h0_in_place(schedule):
    """h0 may be last_state itself: the state is continued in place."""
    if schedule == "balanced":
        w, kw = synth.fwd_inputs(6, 1000, 4096, 16, seed=46), dict(workspace=True, force=Force(nseg=0))
    else:
        w = synth.fwd_inputs(2, 900, 64, 16, seed=46)
        kw = {"lane": dict(workspace=False, force=Force(0, 4, 1, nseg=0)),
              "seg": dict(workspace=False, force=Force(1, 0, 1, nseg=0)),
              "timesplit": dict(workspace=True, force=Force(nseg=5))}[schedule]
    h0 = synth.initial_state(w.batch, w.Dm, w.N, seed=46)
    y, last = gpu(w, h0, in_place=True, **kw)
    ry, rlast, mag = ref(w, h0)
    assert_fwd_close("f32", y, ry, mag, last, rlast, what=f"in place {schedule}")


def test_h0_L_zero_copies_state():
    h0 = torch.from_numpy(synth.initial_state(2, 24, 16, seed=47)).cuda()
    last = torch.full((2, 24, 16), float("nan"), device="cuda")
    e = torch.empty((2, 0, 24), device="cuda")
    bc = torch.empty((2, 0, 16), device="cuda")
    ss.ss_fwd(e, e, None, torch.zeros(24, 16, device="cuda"), bc, bc, last_state=last, h0=h0)
    torch.cuda.synchronize()
    assert torch.equal(last, h0)


def test_h0_rejects_overlap_and_misalignment():
    w = synth.fwd_inputs(1, 64, 32, 16, seed=48)
    t = dev(w)
    lib = ss.lib()
    s = ss.FwdStrides(ss.SS_F32, 64 * 32, 32, 64 * 32, 32, 64 * 32, 32, 64 * 32, 32, 64 * 16, 16, 64 * 16, 16)
    y = torch.empty((1, 64, 32), device="cuda")
    big = torch.zeros(2 * 32 * 16 + 8, device="cuda")
    last = big[: 32 * 16]

    def call(h0_ptr, y_ptr=None, last_ptr=None):
        return lib.ss_fwd_h0(t["u"].data_ptr(), t["delta_raw"].data_ptr(), t["delta_bias"].data_ptr(),
                             t["A_log"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(), t["D"].data_ptr(),
                             t["z"].data_ptr(), y_ptr or y.data_ptr(), last_ptr or last.data_ptr(), h0_ptr,
                             1, 64, 32, 16, ctypes.byref(s), None, 0, None)
    assert call(big[16:].data_ptr()) == 1                      # overlaps last_state, not equal
    assert call(y.data_ptr()) == 1                             # overlaps y
    assert call(big.data_ptr() + 2) == 3                       # not 4-byte aligned
    assert call(big[32 * 16:].data_ptr()) == 0                 # disjoint
    assert call(last.data_ptr()) == 0                          # in place


# ------------------------------------------------------------------ the time-split schedule

@pytest.mark.parametrize("nseg", [2, 3, 7, 64])
@pytest.mark.parametrize("with_h0", [False, True], ids=["zero", "h0"])
def test_timesplit_forced_segments(nseg, with_h0):
    w = synth.fwd_inputs(2, 1000, 96, 16, seed=50 + nseg)
    h0 = synth.initial_state(2, 96, 16, seed=50) if with_h0 else None
    check(w, h0, workspace=True, force=Force(nseg=nseg))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N,lpc", [(16, 4), (16, 2), (16, 1), (8, 2), (8, 1), (4, 1)])
def test_timesplit_state_counts_and_lanes(io, N, lpc):
    """The time split is TMA-fed, so N is a kernel state width (4, 8 or 16)."""
    if io == "bf16" and N == 4:
        pytest.skip("bf16 B/C rows of 4 states are 8 bytes, below the 16-byte TMA row minimum")
    w = synth.fwd_inputs(1, 777, 72, N, io=io, seed=60 + N)
    check(w, synth.initial_state(1, 72, N, seed=60), workspace=True, force=Force(0, lpc, 1, nseg=4))


@pytest.mark.parametrize("N", [5, 12])
def test_timesplit_not_used_without_tma(N):
    """N below the kernel's state width cannot use TMA tiles: a forced split falls back to the
    plain-load per-tile schedule, same result."""
    w = synth.fwd_inputs(1, 500, 40, N, seed=61 + N)
    check(w, synth.initial_state(1, 40, N, seed=61), workspace=True, force=Force(nseg=4))


@pytest.mark.parametrize("L", [65, 128, 129, 1000, 4097])
def test_timesplit_ragged_lengths(L):
    w = synth.fwd_inputs(1, L, 48, 16, seed=70 + L % 97)
    check(w, synth.initial_state(1, 48, 16, seed=70), workspace=True, force=Force(nseg=3))


def test_timesplit_is_chosen_for_few_tiles_and_matches_plain():
    """Automatic choice: one long sequence over few channels takes the time split with a
    workspace; it matches the oracle and, up to rounding, the plain schedule."""
    w = synth.fwd_inputs(1, 8192, 256, 16, seed=71)
    assert ss.ss_fwd_workspace_size(1, 8192, 256, 16) > 0
    y_ws, l_ws = check(w, workspace=True)
    y_pl, l_pl = gpu(w, workspace=False)
    assert rel_l2(y_ws, y_pl) <= FP32_REL_L2
    assert rel_l2(l_ws, l_pl) <= FP32_REL_L2


def test_timesplit_long32k_sampled_rows():
    """The long-sequence workload (batch 1, L 32768, Dm 1536, N 16) in the launch the
    workspace path makes, checked on sampled channels against the oracle."""
    w = synth.config("long32k")
    t = dev(w)
    last = torch.empty((1, 1536, 16), device="cuda")
    y = ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                  last_state=last, workspace=True)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 31, 32, 500, 767, 1024, 1535])
    a = w.arrays
    ry, rlast, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                   a["z"], rows=rows)
    yh = to_host(y)[0][:, rows].T                     # [rows, L]
    assert_fwd_close("f32", yh, ry, mag, to_host(last)[0][rows], rlast, what="long32k time-split")


def test_timesplit_small_workspace_uses_fewer_segments():
    """A workspace too small for the planned segments gives fewer (same result); one too
    small for two runs the per-tile schedule."""
    w = synth.fwd_inputs(1, 4000, 64, 16, seed=72)
    t = dev(w)
    lib = ss.lib()
    s = ss.FwdStrides(ss.SS_F32, 4000 * 64, 64, 4000 * 64, 64, 4000 * 64, 64, 4000 * 64, 64, 4000 * 16, 16,
                      4000 * 16, 16)
    need = ss.ss_fwd_workspace_size(1, 4000, 64, 16)
    assert need > 0
    ry, rlast, mag = ref(w)
    for nbytes in (need, need // 2, 64 * 16 * 4 * 2 + 64 * 4 + 256, 100):
        ws = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device="cuda")
        y = torch.empty((1, 4000, 64), device="cuda")
        last = torch.empty((1, 64, 16), device="cuda")
        st = lib.ss_fwd_ws(t["u"].data_ptr(), t["delta_raw"].data_ptr(), t["delta_bias"].data_ptr(),
                           t["A_log"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(), t["D"].data_ptr(),
                           t["z"].data_ptr(), y.data_ptr(), last.data_ptr(), 1, 4000, 64, 16, ctypes.byref(s),
                           ws.data_ptr(), nbytes, None)
        assert st == 0, nbytes
        torch.cuda.synchronize()
        assert_fwd_close("f32", to_host(y), ry, mag, to_host(last), rlast, what=f"ws {nbytes} B")
