"""Shared test helpers: error metrics and host<->device marshalling of synthetic inputs."""
import numpy as np

# Accuracy targets: fp32 I/O max relative error 1e-4 and relative L2 1e-5; bf16 I/O with
# fp32 state relative L2 5e-3.  The relative error of one output is taken against
# |y_ref| + m, m being the size of the terms summed into it (oracle's `mag`), because
# y itself can cancel to ~0 (silu(z) ~ 0 or C·h ~ -D·u).
FP32_MAX_REL = 1e-4
FP32_REL_L2 = 1e-5
BF16_REL_L2 = 5e-3
STATE_REL_L2 = 1e-5


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return num / den if den > 0 else num


def max_rel(got, ref, mag):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref) + np.asarray(mag, np.float64)
    err = np.abs(got - ref)
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(den > 0, err / den, err)
    return float(r.max()) if r.size else 0.0


def plain_max_rel(got, ref):
    """max_i |e_i| / max_i |y_ref,i|: the largest error against the output's scale (recorded
    beside the condition-aware max_rel, which divides each error by its own term sizes)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    return err / scale if scale > 0 else err


# Every assert_fwd_close call appends (what, io, rel-L2, max-rel, plain max-rel) here; conftest
# prints the worst of each at the end of the session.
RECORDED = []


def assert_fwd_close(io, y, ref_y, mag, last=None, ref_last=None, what=""):
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    e2 = rel_l2(y, ref_y)
    RECORDED.append((what, io, e2, max_rel(y, ref_y, mag) if io == "f32" else float("nan"),
                     plain_max_rel(y, ref_y)))
    if io == "bf16":
        assert e2 <= BF16_REL_L2, f"{what}: y rel-L2 {e2:.3e} > {BF16_REL_L2}"
    else:
        mr = max_rel(y, ref_y, mag)
        assert mr <= FP32_MAX_REL, f"{what}: y max-rel {mr:.3e} > {FP32_MAX_REL}"
        assert e2 <= FP32_REL_L2, f"{what}: y rel-L2 {e2:.3e} > {FP32_REL_L2}"
    if last is not None:
        el = rel_l2(last, ref_last)
        tol = STATE_REL_L2 if io == "f32" else 1e-4
        assert el <= tol, f"{what}: last_state rel-L2 {el:.3e} > {tol}"


def to_dev(arr, io, device="cuda"):
    """float32 numpy array holding exact io values -> torch tensor of the io dtype."""
    import torch
    if arr is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(device)
    return t.to(torch.bfloat16) if io == "bf16" else t


def f32dev(arr, device="cuda"):
    import torch
    return None if arr is None else torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(device)


def to_host(t):
    return t.float().cpu().numpy().astype(np.float64)
