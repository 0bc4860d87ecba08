"""Parity of the CUDA decode step (through the C ABI) with the fp64 oracle, and the
decode == scan identities between the two entry points."""
import ctypes

import numpy as np
import pytest

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


def gpu_step(w, state_dev=None):
    a = w.arrays
    io = w.io
    st = f32dev(a["state"]) if state_dev is None else state_dev
    y = ss.ss_step(st, to_dev(a["x"], io), to_dev(a["delta_raw"], io), f32dev(a["delta_bias"]),
                   f32dev(a["A_log"]), to_dev(a["B"], io), to_dev(a["C"], io), f32dev(a["D"]),
                   to_dev(a["z"], io))
    torch.cuda.synchronize()
    return to_host(y), st


def oracle_step(w):
    a = w.arrays
    return oracle.ss_step(a["state"], a["x"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"],
                          a["C"], a["D"], a["z"])


def check_step(w):
    y, st = gpu_step(w)
    ry, rst, mag = oracle_step(w)
    assert_fwd_close(w.io, y, ry, mag, to_host(st), rst, what=f"step {w.name} {w.io} N={w.N}")


def test_decode_workload_one_layer():
    check_step(synth.config("decode1p4b"))


def test_decode_workload_48_layers():
    """Every one of the 48 layers' distinct states and inputs, stepped once in order."""
    for layer in range(48):
        check_step(synth.step_inputs(64, 4096, 16, seed=4, layer=layer))


@pytest.mark.parametrize("N", [1, 3, 4, 5, 8, 11, 16])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_state_counts(N, io):
    check_step(synth.step_inputs(5, 77, N, io=io, seed=40 + N, with_bias=True))


def test_step_without_gate_and_skip():
    w = synth.step_inputs(4, 64, 16, seed=41)
    w.arrays["z"] = None
    w.arrays["D"] = None
    check_step(w)


def test_step_strided_state():
    """State as a view with padded per-channel and per-batch strides."""
    w = synth.step_inputs(3, 40, 16, seed=42)
    big = torch.zeros((3, 41, 20), device="cuda")
    big[:, :40, :16] = f32dev(w.arrays["state"])
    view = big[:, :40, :16]
    y, _ = gpu_step(w, state_dev=view)
    ry, rst, mag = oracle_step(w)
    assert_fwd_close("f32", y, ry, mag, to_host(view), rst, what="strided state")
    assert torch.all(big[:, 40, :] == 0) and torch.all(big[:, :, 16:] == 0)


def _fwd_dev(w):
    a = w.arrays
    io = w.io
    return dict(u=to_dev(a["u"], io), delta_raw=to_dev(a["delta_raw"], io), z=to_dev(a["z"], io),
                B=to_dev(a["B"], io), C=to_dev(a["C"], io), A_log=f32dev(a["A_log"]),
                D=f32dev(a["D"]), delta_bias=f32dev(a["delta_bias"]))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_iterated_step_equals_forward(io):
    """ss_step run L times from h = 0 reproduces ss_fwd's y and last_state."""
    w = synth.fwd_inputs(2, 120, 48, 16, io=io, seed=43)
    t = _fwd_dev(w)
    last = torch.empty((2, 48, 16), device="cuda")
    y_fwd = ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"],
                      t["z"], last_state=last)
    state = torch.zeros((2, 48, 16), device="cuda")
    ys = []
    for k in range(120):
        ys.append(ss.ss_step(state, t["u"][:, k], t["delta_raw"][:, k], t["delta_bias"], t["A_log"],
                             t["B"][:, k], t["C"][:, k], t["D"], t["z"][:, k]))
    torch.cuda.synchronize()
    y_step = torch.stack(ys, dim=1)
    ry, rlast, mag = oracle.ss_fwd(*(w.arrays[k] for k in ("u", "delta_raw", "delta_bias", "A_log",
                                                            "B", "C", "D", "z")))
    assert_fwd_close(io, to_host(y_step), ry, mag, to_host(state), rlast, what="iterated step")
    tol = 1e-5 if io == "f32" else 2e-2
    assert rel_l2(to_host(y_step), to_host(y_fwd)) < tol
    assert rel_l2(to_host(state), to_host(last)) < 1e-5


def test_prefill_then_decode_equals_forward():
    """ss_fwd over a prefix, its last_state handed to ss_step for the rest, equals ss_fwd over
    the whole sequence."""
    w = synth.fwd_inputs(2, 300, 64, 16, seed=44)
    t = _fwd_dev(w)
    k = 211
    state = torch.empty((2, 64, 16), device="cuda")
    ss.ss_fwd(t["u"][:, :k], t["delta_raw"][:, :k], t["delta_bias"], t["A_log"], t["B"][:, :k],
              t["C"][:, :k], t["D"], t["z"][:, :k], last_state=state)
    ys = [ss.ss_step(state, t["u"][:, j], t["delta_raw"][:, j], t["delta_bias"], t["A_log"],
                     t["B"][:, j], t["C"][:, j], t["D"], t["z"][:, j]) for j in range(k, 300)]
    torch.cuda.synchronize()
    ry, rlast, mag = oracle.ss_fwd(*(w.arrays[n] for n in ("u", "delta_raw", "delta_bias", "A_log",
                                                            "B", "C", "D", "z")))
    assert_fwd_close("f32", to_host(torch.stack(ys, 1)), ry[:, k:], mag[:, k:], to_host(state), rlast,
                     what="prefill+decode")


def _layer_tensors(w, state_dev=None):
    a = w.arrays
    io = w.io
    return {"state": f32dev(a["state"]) if state_dev is None else state_dev, "x": to_dev(a["x"], io),
            "delta_raw": to_dev(a["delta_raw"], io), "delta_bias": f32dev(a["delta_bias"]),
            "A_log": f32dev(a["A_log"]), "B": to_dev(a["B"], io), "C": to_dev(a["C"], io), "D": f32dev(a["D"]),
            "z": to_dev(a["z"], io)}


def test_step_layers_decode_workload_48_layers():
    """All 48 layers of the decode workload in one ss_step_layers launch: every layer's y and
    updated state against the oracle, and bit for bit against 48 ss_step calls."""
    ws = [synth.step_inputs(64, 4096, 16, seed=4, layer=layer) for layer in range(48)]
    batched = [_layer_tensors(w) for w in ws]
    ys = ss.ss_step_layers(batched)
    torch.cuda.synchronize()
    for w, L, y in zip(ws, batched, ys):
        ry, rst, mag = oracle_step(w)
        assert_fwd_close("f32", to_host(y), ry, mag, to_host(L["state"]), rst, what=f"layers {w.name}")
        y1, st1 = gpu_step(w)
        np.testing.assert_array_equal(to_host(y), y1)
        np.testing.assert_array_equal(to_host(L["state"]), to_host(st1))


@pytest.mark.parametrize("N", [4, 5, 16])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_layers_shapes(N, io):
    """A few layers of ragged sizes (the vector path at N = 4, 16; the scalar one at N = 5)."""
    ws = [synth.step_inputs(3, 77, N, io=io, seed=60 + N + k, with_bias=True) for k in range(5)]
    batched = [_layer_tensors(w) for w in ws]
    ys = ss.ss_step_layers(batched)
    torch.cuda.synchronize()
    for w, L, y in zip(ws, batched, ys):
        ry, rst, mag = oracle_step(w)
        assert_fwd_close(io, to_host(y), ry, mag, to_host(L["state"]), rst, what=f"layers N={N} {io}")


def test_step_layers_rejects_shared_outputs_and_too_many_layers():
    w = synth.step_inputs(2, 32, 16, seed=70)
    a, b = _layer_tensors(w), _layer_tensors(w)
    b["state"] = a["state"]                     # two layers writing one state
    with pytest.raises(ss.SelscanError):
        ss.ss_step_layers([a, b])
    c = _layer_tensors(w)
    c["x"] = a["state"].view(-1)[: 2 * 32].view(2, 32)   # a layer reading another's state
    with pytest.raises(ss.SelscanError):
        ss.ss_step_layers([a, c])
    many = [_layer_tensors(w) for _ in range(129)]
    with pytest.raises(ss.SelscanError):
        ss.ss_step_layers(many)
    assert ss.ss_step_layers([]) == []


def _force_layers_path(v):
    f = ss.lib().ss__force_step_layers_path
    f.argtypes = [ctypes.c_int]
    f.restype = ctypes.c_int
    return f(v)


def _layers_run(ws, path):
    """ss_step_layers over the layers of `ws` on a forced kernel (0 per-block, 1 staged)."""
    batched = [_layer_tensors(w) for w in ws]
    _force_layers_path(path)
    try:
        ys = ss.ss_step_layers(batched)
        torch.cuda.synchronize()
    finally:
        _force_layers_path(-1)
    return [to_host(y) for y in ys], [to_host(L["state"]) for L in batched]


def test_step_layers_staged_equals_block_kernel_on_decode_workload():
    """The staged kernel (each warp's contiguous range of 32-row units streamed through its own
    ring of bulk-copied stages) computes every row with the per-block kernel's arithmetic: the
    same y and states bit for bit on 12 layers of the decode workload, and the oracle's."""
    ws = [synth.step_inputs(64, 4096, 16, seed=4, layer=layer) for layer in range(12)]
    y1, s1 = _layers_run(ws, 1)
    y0, s0 = _layers_run(ws, 0)
    for w, a, b, sa, sb in zip(ws, y1, y0, s1, s0):
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(sa, sb)
    for w, y, st in list(zip(ws, y1, s1))[:3]:
        ry, rst, mag = oracle_step(w)
        assert_fwd_close("f32", y, ry, mag, st, rst, what=f"staged {w.name}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(with_z=True, with_bias=True), dict(with_z=False, with_bias=False)])
def test_step_layers_staged_ranges_cross_layers_and_rows(io, opts):
    """7 layers of batch 5 and 96 channels (three 32-row units a batch row, one unit a warp;
    the decode-workload test above gives each warp a range of about 50 units across batch rows
    and layers), with and without the gate and the bias, and without D on some layers."""
    ws = [synth.step_inputs(5, 96, 16, io=io, seed=80 + k, **opts) for k in range(7)]
    for k in (1, 4):
        ws[k].arrays["D"] = None
    y1, s1 = _layers_run(ws, 1)
    for w, y, st in zip(ws, y1, s1):
        ry, rst, mag = oracle_step(w)
        assert_fwd_close(io, y, ry, mag, st, rst, what=f"staged ragged {io} {opts}")
    y0, s0 = _layers_run(ws, 0)
    for a, b, sa, sb in zip(y1, y0, s1, s0):
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(sa, sb)


def test_step_layers_staged_refused_where_it_cannot_run():
    """Channels that are not whole 32-row units, or 8 states: the staged kernel is refused when
    forced (no silent substitute), and the automatic choice runs the per-block kernel."""
    for Dm, N in ((77, 16), (64, 8)):
        ws = [synth.step_inputs(3, Dm, N, seed=90 + Dm, with_bias=True) for _ in range(2)]
        with pytest.raises(ss.SelscanError):
            _layers_run(ws, 1)
        ys, sts = _layers_run(ws, -1)
        for w, y, st in zip(ws, ys, sts):
            ry, rst, mag = oracle_step(w)
            assert_fwd_close("f32", y, ry, mag, st, rst, what=f"auto Dm={Dm} N={N}")


def test_step_single_layer_staged_equals_block_kernel():
    """ss_step on one layer of the decode workload takes the staged kernel too (a table of one
    layer): bit for bit the per-block kernel's y and state."""
    w = synth.step_inputs(64, 4096, 16, seed=4, layer=7)
    out = {}
    for path in (1, 0):
        _force_layers_path(path)
        try:
            out[path] = gpu_step(w)
        finally:
            _force_layers_path(-1)
    np.testing.assert_array_equal(out[1][0], out[0][0])
    np.testing.assert_array_equal(to_host(out[1][1]), to_host(out[0][1]))


def test_step_layers_at_the_layer_limit():
    """128 layers (the most one call takes) of batch 3 and 64 channels through the staged kernel,
    each against the oracle."""
    ws = [synth.step_inputs(3, 64, 16, seed=300 + k, with_bias=bool(k % 2)) for k in range(128)]
    ys, sts = _layers_run(ws, 1)
    for w, y, st in zip(ws, ys, sts):
        ry, rst, mag = oracle_step(w)
        assert_fwd_close("f32", y, ry, mag, st, rst, what=f"128 layers {w.seed}")
