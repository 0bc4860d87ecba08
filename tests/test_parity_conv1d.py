"""Parity of the CUDA causal depthwise conv1d (through the C ABI) with the fp64 oracle."""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import BF16_REL_L2, rel_l2, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CONV_MAX_REL = 1e-5      # fp32: 4 fused multiply-adds and an SFU silu per output
CONV_REL_L2 = 1e-6


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def inputs(seed, batch, L, Dm, io="f32"):
    g = synth.rng_for(seed, 9)
    x = g.standard_normal((batch, L, Dm), dtype=np.float32)
    if io == "bf16":
        x = synth.round_bf16(x)
    w = (0.5 * g.standard_normal((Dm, 4), dtype=np.float32)).astype(np.float32)
    bias = (0.1 * g.standard_normal(Dm, dtype=np.float32)).astype(np.float32)
    win = g.standard_normal((batch, Dm, 3), dtype=np.float32)
    if io == "bf16":
        win = synth.round_bf16(win)
    return x, w, bias, win


def check(io, y, x, w, bias, win, silu, what, win_out=None):
    ref, wref = oracle.conv1d(x, w, bias, window=win, act=silu)
    mag, _ = oracle.conv1d(np.abs(x), np.abs(w), None if bias is None else np.abs(bias),
                           window=None if win is None else np.abs(win), act=False)
    assert np.all(np.isfinite(y)), what
    if io == "bf16":
        assert rel_l2(y, ref) <= BF16_REL_L2, f"{what}: rel-L2 {rel_l2(y, ref):.3e}"
    else:
        mr = float(np.max(np.abs(y - ref) / (np.abs(ref) + mag + 1e-30)))
        assert mr <= CONV_MAX_REL, f"{what}: max-rel {mr:.3e}"
        assert rel_l2(y, ref) <= CONV_REL_L2, f"{what}: rel-L2 {rel_l2(y, ref):.3e}"
    if win_out is not None:
        np.testing.assert_array_equal(win_out, wref.astype(np.float32).astype(np.float64))


def run(x, w, bias, win, silu, io="f32", in_place=False, want_win=True):
    xd = to_dev(x, io)
    wd = torch.from_numpy(w).cuda()
    bd = None if bias is None else torch.from_numpy(bias).cuda()
    wi = None if win is None else torch.from_numpy(np.ascontiguousarray(win, np.float32)).cuda()
    wo = None
    if want_win:
        wo = wi if (in_place and wi is not None) else torch.full((x.shape[0], x.shape[2], 3), float("nan"), device="cuda")
    y = ss.ss_conv1d(xd, wd, bd, window_in=wi, window_out=wo, silu=silu)
    torch.cuda.synchronize()
    return to_host(y), (None if wo is None else to_host(wo))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 2, 3, 4, 63, 64, 65, 200, 1000])
def test_conv1d_lengths(io, L):
    x, w, bias, win = inputs(L, 2, L, 96, io)
    for silu in (True, False):
        y, wo = run(x, w, bias, win, silu, io)
        check(io, y, x, w, bias, win, silu, f"L={L} {io} silu={silu}", wo)


@pytest.mark.parametrize("Dm", [1, 3, 4, 5, 127, 128, 513, 1000])
def test_conv1d_channel_counts(Dm):
    """Dm % 4 != 0 takes the scalar path; every Dm ends in a partial block."""
    x, w, bias, win = inputs(100 + Dm, 3, 77, Dm)
    y, wo = run(x, w, bias, win, True)
    check("f32", y, x, w, bias, win, True, f"Dm={Dm}", wo)


@pytest.mark.parametrize("opts", ["no_bias", "no_window", "no_window_out", "none"])
def test_conv1d_optional_inputs(opts):
    x, w, bias, win = inputs(7, 2, 150, 64)
    if opts in ("no_bias", "none"):
        bias = None
    if opts in ("no_window", "none"):
        win = None
    y, wo = run(x, w, bias, win, True, want_win=opts != "no_window_out")
    check("f32", y, x, w, bias, win, True, opts, wo)


def test_conv1d_strided_input():
    """x as the first half of a wider [batch, L, 2*Dm] tensor (the in_proj output split)."""
    x, w, bias, win = inputs(8, 2, 130, 64)
    wide = np.concatenate([x, np.zeros_like(x)], axis=2)
    wd = torch.from_numpy(wide).cuda()
    xv = wd[:, :, :64]
    y = ss.ss_conv1d(xv, torch.from_numpy(w).cuda(), torch.from_numpy(bias).cuda(),
                     window_in=torch.from_numpy(win).cuda(), silu=True)
    torch.cuda.synchronize()
    check("f32", to_host(y), x, w, bias, win, True, "strided")


@pytest.mark.parametrize("k", [1, 2, 3, 64, 100, 257])
def test_conv1d_split_across_calls_in_place(k):
    """Chunked prefill with one window buffer updated in place equals one call."""
    x, w, bias, win = inputs(9, 2, 300, 128)
    y_full, wo_full = run(x, w, bias, win, True)
    y1, wbuf = run(x[:, :k], w, bias, win, True, in_place=True)
    y2, wbuf2 = run(x[:, k:], w, bias, wbuf, True, in_place=True)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y_full, rtol=0, atol=0)
    np.testing.assert_array_equal(wbuf2, wo_full)


def test_conv1d_decode_steps_equal_prefill():
    """L = 1 calls (decode) with the window updated in place reproduce the prefill output."""
    x, w, bias, win = inputs(10, 3, 20, 256)
    y_full, _ = run(x, w, bias, win, True)
    wbuf = torch.from_numpy(win).cuda()
    wd, bd = torch.from_numpy(w).cuda(), torch.from_numpy(bias).cuda()
    outs = []
    for t in range(20):
        xt = torch.from_numpy(np.ascontiguousarray(x[:, t:t + 1])).cuda()
        outs.append(to_host(ss.ss_conv1d(xt, wd, bd, window_in=wbuf, window_out=wbuf, silu=True)))
    torch.cuda.synchronize()
    np.testing.assert_allclose(np.concatenate(outs, axis=1), y_full, rtol=0, atol=0)


def test_conv1d_full_size_130m_shape():
    """The conv1d input of the 130m-shaped layer (batch 8, L 2048, Dm 1536), fp32 and bf16."""
    for io in ("f32", "bf16"):
        x, w, bias, win = inputs(11, 8, 2048, 1536, io)
        y, wo = run(x, w, bias, None, True, io)
        check(io, y, x, w, bias, None, True, f"130m shape {io}", wo)


def test_conv1d_L_zero_copies_window():
    win = torch.randn(2, 16, 3, device="cuda")
    wout = torch.full((2, 16, 3), float("nan"), device="cuda")
    e = torch.empty((2, 0, 16), device="cuda")
    ss.ss_conv1d(e, torch.zeros(16, 4, device="cuda"), window_in=win, window_out=wout)
    torch.cuda.synchronize()
    assert torch.equal(win, wout)


def test_conv1d_rejects_overlap_and_misalignment():
    lib = ss.lib()
    x = torch.randn(1, 64, 32, device="cuda")
    w = torch.randn(32, 4, device="cuda")
    out = torch.empty(1, 64, 32, device="cuda")
    big = torch.zeros(200, device="cuda")
    s = ss.ConvStrides(ss.SS_F32, 64 * 32, 32, 64 * 32, 32)

    def call(xp, outp, wi=None, wo=None):
        return lib.ss_conv1d(xp, w.data_ptr(), None, outp, wi, wo, 1, 64, 32, 1, ctypes.byref(s), None)
    assert call(x.data_ptr(), x.data_ptr()) == 1                       # out overlaps x
    assert call(x.data_ptr(), out.data_ptr(), None, x.data_ptr()) == 1  # window_out overlaps x
    assert call(x.data_ptr(), out.data_ptr(), big.data_ptr(), big[8:].data_ptr()) == 1   # windows overlap
    assert call(x.data_ptr() + 2, out.data_ptr()) == 3                  # misaligned x
    assert call(x.data_ptr(), out.data_ptr(), big.data_ptr(), big.data_ptr()) == 0       # in place
    torch.cuda.synchronize()


@pytest.mark.parametrize("steps", [3, 7, 16, 41, 128, 300])
def test_conv1d_segment_length_invariance(steps):
    """The steps each thread takes (chosen per call to fill whole waves; forced here) change
    nothing: the same outputs and window bit for bit, with and without the incoming window."""
    f = ss.lib().ss__force_conv_segment
    f.argtypes = [ctypes.c_int]
    x, w, bias, win = inputs(20 + steps, 3, 1000, 608)
    ref = run(x, w, bias, win, True)
    f(steps)
    try:
        got = run(x, w, bias, win, True)
        got0 = run(x, w, bias, None, False)
    finally:
        f(0)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    check("f32", got[0], x, w, bias, win, True, f"segment {steps}", got[1])
    check("f32", got0[0], x, w, bias, None, False, f"segment {steps} no window", got0[1])
