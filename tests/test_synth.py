"""The seeded input generator, against the recipe the workloads are stated with: the shapes
of the five workloads, reproducibility, the value distributions of each recipe, and the
bf16 rounding (nearest, ties to even) checked against a separate definition.  CPU only."""
import numpy as np
import pytest

from selective_state_space_scan_gb300 import synth


def test_same_seed_same_arrays_and_seeds_differ():
    a = synth.fwd_inputs(2, 33, 20, 5, seed=7).arrays
    b = synth.fwd_inputs(2, 33, 20, 5, seed=7).arrays
    c = synth.fwd_inputs(2, 33, 20, 5, seed=8).arrays
    for k in ("u", "delta_raw", "z", "B", "C", "delta_bias", "D", "A_log"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("u", "delta_raw", "z", "B", "C", "delta_bias", "D"):
        assert not np.array_equal(a[k], c[k]), k
    # the decode layers and the initial state draw from streams of their own
    s0, s1 = synth.step_inputs(4, 8, 4, layer=0), synth.step_inputs(4, 8, 4, layer=1)
    assert not np.array_equal(s0.arrays["state"], s1.arrays["state"])
    assert not np.array_equal(synth.initial_state(2, 20, 5, seed=7).ravel()[:10], a["u"].ravel()[:10])


def test_workload_shapes():
    want = {"tiny": (1, 64, 16, 4, "f32"), "mamba130m": (8, 2048, 1536, 16, "f32"),
            "long32k": (1, 32768, 1536, 16, "f32"), "mamba2p8b_bf16": (4, 8192, 5120, 16, "bf16"),
            "decode1p4b": (64, 1, 4096, 16, "f32")}
    for name, (batch, L, Dm, N, io) in want.items():
        c = synth.CONFIGS[name]
        assert (c["batch"], c["L"], c["Dm"], c["N"], c["io"]) == (batch, L, Dm, N, io), name
    assert [synth.CONFIGS[n]["seed"] for n in want] == [0, 1, 2, 3, 4]
    t = synth.config("tiny")
    assert t.arrays["u"].shape == (1, 64, 16) and t.arrays["B"].shape == (1, 64, 4)
    assert t.arrays["A_log"].shape == (16, 4) and t.arrays["D"].shape == (16,)
    d = synth.config("decode1p4b")
    assert d.arrays["state"].shape == (64, 4096, 16) and d.arrays["x"].shape == (64, 4096)
    assert d.arrays["B"].shape == (64, 16)


def _near(x, mean, sd, k=6.0):
    """Sample mean within k standard errors of the mean, sample sd within k of its own."""
    x = np.asarray(x, np.float64).ravel()
    se = sd / np.sqrt(x.size)
    assert abs(x.mean() - mean) <= k * se, (x.mean(), mean)
    assert abs(x.std() - sd) <= k * sd / np.sqrt(2 * x.size), (x.std(), sd)


def test_mamba_recipe_distributions():
    a = synth.fwd_inputs(2, 512, 256, 16, seed=5).arrays
    _near(a["u"], 0.0, 1.0)
    _near(a["z"], 0.0, 1.0)
    _near(a["delta_raw"], -4.0, 1.0)
    _near(a["B"], 0.0, 1.0)
    _near(a["C"], 0.0, 1.0)
    bias = a["delta_bias"].astype(np.float64)
    assert bias.min() >= -1.0 and bias.max() <= 0.0
    _near(bias, -0.5, np.sqrt(1 / 12))                    # U(-1, 0)
    _near(a["D"], 1.0, 0.1)                               # N(1, 0.1): 0.1 is the sd
    want = np.log(np.arange(1, 17, dtype=np.float64)).astype(np.float32)
    assert np.array_equal(a["A_log"], np.tile(want, (256, 1)))   # the same row for every channel


def test_tiny_and_decode_recipes():
    t = synth.config("tiny").arrays
    assert np.all(t["delta_bias"] == np.float32(0.1)) and np.all(t["D"] == 1.0)
    assert np.array_equal(t["A_log"][0], np.log(np.arange(1, 5)).astype(np.float32))
    big = synth.fwd_inputs(4, 256, 64, 4, dist="tiny", seed=9).arrays
    _near(big["delta_raw"], 0.0, 1.0)
    d = synth.step_inputs(64, 512, 16, seed=4).arrays
    _near(d["state"], 0.0, 0.5)                           # h ~ N(0, 0.5): 0.5 is the sd
    _near(d["x"], 0.0, 1.0)
    assert d["delta_bias"] is None and np.all(d["D"] == 1.0)
    _near(synth.initial_state(8, 256, 16, seed=1), 0.0, 0.5)


def _bf16_reference(x):
    """Nearest bfloat16 of each float32 (ties to the even significand), from the two bf16
    neighbours computed in float64: an independent restatement of round-to-nearest-even."""
    out = np.empty(x.shape, np.uint16)
    for i, v in enumerate(x.ravel()):
        bits = int(np.float32(v).view(np.uint32))
        lo = bits >> 16                                    # truncation toward zero (same sign)
        hi = lo + 1                                        # the next bf16 away from zero
        f = lambda b: float(np.uint32(b << 16).view(np.float32))
        dlo, dhi = abs(float(v) - f(lo)), abs(f(hi) - float(v))
        if dlo < dhi or (dlo == dhi and lo % 2 == 0):
            out.ravel()[i] = lo
        else:
            out.ravel()[i] = hi
    return out


def test_bf16_rounding_is_nearest_even():
    g = np.random.default_rng(0)
    x = (g.standard_normal(4000) * np.exp2(g.integers(-20, 20, 4000))).astype(np.float32)
    # exact ties: a bf16 value plus half its last place, and a few near-ties
    base = synth.round_bf16(g.standard_normal(200).astype(np.float32)).view(np.uint32)
    ties = (base + np.uint32(0x8000)).view(np.float32)
    near = np.concatenate([(base + np.uint32(0x7FFF)).view(np.float32), (base + np.uint32(0x8001)).view(np.float32)])
    for arr in (x, ties, near, np.array([0.0, -0.0, 1.0, -1.5, 3.0e38], np.float32)):
        assert np.array_equal(synth.bf16_bits(arr), _bf16_reference(arr))


def test_bf16_workload_holds_exact_bf16_values():
    w = synth.fwd_inputs(1, 40, 24, 8, io="bf16", seed=3)
    for k in ("u", "delta_raw", "z", "B", "C"):
        assert np.all((w.arrays[k].view(np.uint32) & 0xFFFF) == 0), k
    f32 = synth.fwd_inputs(1, 40, 24, 8, io="f32", seed=3)
    for k in ("delta_bias", "D", "A_log"):                 # parameters stay fp32
        assert np.array_equal(w.arrays[k], f32.arrays[k]), k
    assert np.array_equal(w.arrays["u"], synth.round_bf16(f32.arrays["u"]))


@pytest.mark.parametrize("bad", ["gauss", ""])
def test_unknown_recipe_is_refused(bad):
    with pytest.raises(ValueError):
        synth.fwd_inputs(1, 4, 4, 4, dist=bad)
