"""fp64 CPU oracle for the selective scan — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python binding)
never imports it, and it imports nothing from the product.

The arithmetic lives in ``selscan_oracle.c`` (plain sequential fp64 loops); this
module only marshals numpy arrays into it.  See that file's header for the passages
each function follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_ss_fwd_rows.argtypes = [f32p] * 8 + [f64p, i64p, i64, f64p, f64p, f64p, i64, i64, i64, i64]
    lib.oracle_ss_fwd_rows.restype = ctypes.c_int
    lib.oracle_ss_fwd_dtproj_rows.argtypes = [f32p] * 3 + [i64] + [f32p] * 6 + [f64p, i64p, i64, f64p, f64p, f64p,
                                                                               i64, i64, i64, i64]
    lib.oracle_ss_fwd_dtproj_rows.restype = ctypes.c_int
    lib.oracle_ss_fwd_chunked.argtypes = [f32p] * 8 + [f64p, f64p, f64p, i64, i64, i64, i64, i64]
    lib.oracle_ss_fwd_chunked.restype = ctypes.c_int
    lib.oracle_ss_step.argtypes = [f64p] + [f32p] * 8 + [f64p, f64p, i64, i64, i64]
    lib.oracle_ss_step.restype = ctypes.c_int
    lib.oracle_ss_bwd.argtypes = [f32p] * 8 + [f64p, f32p, f64p] + [f64p] * 9 + [i64] * 4
    lib.oracle_ss_bwd.restype = ctypes.c_int
    lib.oracle_conv1d.argtypes = [f32p, f32p, f32p, f64p, f64p, f64p, i64, i64, i64, i64, ctypes.c_int]
    lib.oracle_conv1d.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def _f32(a, shape=None, name="array"):
    """Return a C-contiguous float32 view/copy (None stays None)."""
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a, ctype):
    if a is None:
        return ctypes.POINTER(ctype)()
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def softplus(x: float) -> float:
    return float(_load().oracle_softplus(float(x)))


def silu(x: float) -> float:
    return float(_load().oracle_silu(float(x)))


def _h0(h0, batch, Dm, N):
    if h0 is None:
        return None
    h = np.ascontiguousarray(np.asarray(h0, dtype=np.float64))
    if h.shape != (batch, Dm, N):
        raise ValueError(f"h0: expected shape {(batch, Dm, N)}, got {h.shape}")
    return h


def ss_fwd(u, delta_raw, delta_bias, A_log, B, C, D, z, rows=None, h0=None):
    """Sequential fp64 forward scan.

    Shapes: u, delta_raw, z [batch, L, Dm]; B, C [batch, L, N]; A_log [Dm, N];
    D, delta_bias [Dm] (or None).  Inputs are taken as float32 values.  h0 [batch, Dm, N]
    (or None for zeros) is the state before step 0, taken in float64.

    rows=None  -> returns (y [batch, L, Dm], last_state [batch, Dm, N], mag [batch, L, Dm])
    rows=array -> flat indices b*Dm+d; returns (y [nrows, L], last [nrows, N], mag [nrows, L])
    """
    u = _f32(u, name="u")
    if u.ndim != 3:
        raise ValueError("u must be [batch, L, Dm]")
    batch, L, Dm = u.shape
    A_log = _f32(A_log, name="A_log")
    N = A_log.shape[1]
    delta_raw = _f32(delta_raw, (batch, L, Dm), "delta_raw")
    z = _f32(z, (batch, L, Dm), "z")
    B = _f32(B, (batch, L, N), "B")
    C = _f32(C, (batch, L, N), "C")
    D = _f32(D, (Dm,), "D")
    delta_bias = _f32(delta_bias, (Dm,), "delta_bias")
    h0 = _h0(h0, batch, Dm, N)
    if rows is None:
        nrows = batch * Dm
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    y = np.empty((nrows, L), np.float64)
    mag = np.empty((nrows, L), np.float64)
    last = np.empty((nrows, N), np.float64)
    st = _load().oracle_ss_fwd_rows(
        _ptr(u, ctypes.c_float), _ptr(delta_raw, ctypes.c_float), _ptr(delta_bias, ctypes.c_float),
        _ptr(A_log, ctypes.c_float), _ptr(B, ctypes.c_float), _ptr(C, ctypes.c_float),
        _ptr(D, ctypes.c_float), _ptr(z, ctypes.c_float), _ptr(h0, ctypes.c_double),
        _ptr(rows_arr, ctypes.c_int64), nrows,
        _ptr(y, ctypes.c_double), _ptr(mag, ctypes.c_double), _ptr(last, ctypes.c_double),
        batch, L, Dm, N)
    if st != 0:
        raise RuntimeError(f"oracle_ss_fwd_rows failed with status {st}")
    if rows is not None:
        return y, last, mag
    y = y.reshape(batch, Dm, L).transpose(0, 2, 1)
    mag = mag.reshape(batch, Dm, L).transpose(0, 2, 1)
    return np.ascontiguousarray(y), last.reshape(batch, Dm, N), np.ascontiguousarray(mag)


def ss_fwd_dtproj(u, dt_low, W_dt, delta_bias, A_log, B, C, D, z, h0=None):
    """Sequential fp64 forward scan whose pre-softplus time step is the low-rank projection
    delta_raw[b,t,d] = sum_k W_dt[d,k] dt_low[b,t,k], summed in fp64 inside the oracle.
    dt_low [batch, L, R], W_dt [Dm, R]; the rest and the returns as ss_fwd(rows=None)."""
    u = _f32(u, name="u")
    if u.ndim != 3:
        raise ValueError("u must be [batch, L, Dm]")
    batch, L, Dm = u.shape
    W_dt = _f32(W_dt, name="W_dt")
    R = W_dt.shape[1]
    dt_low = _f32(dt_low, (batch, L, R), "dt_low")
    A_log = _f32(A_log, name="A_log")
    N = A_log.shape[1]
    z = _f32(z, (batch, L, Dm), "z")
    B = _f32(B, (batch, L, N), "B")
    C = _f32(C, (batch, L, N), "C")
    D = _f32(D, (Dm,), "D")
    delta_bias = _f32(delta_bias, (Dm,), "delta_bias")
    h0 = _h0(h0, batch, Dm, N)
    nrows = batch * Dm
    y = np.empty((nrows, L), np.float64)
    mag = np.empty((nrows, L), np.float64)
    last = np.empty((nrows, N), np.float64)
    st = _load().oracle_ss_fwd_dtproj_rows(
        _ptr(u, ctypes.c_float), _ptr(dt_low, ctypes.c_float), _ptr(W_dt, ctypes.c_float), R,
        _ptr(delta_bias, ctypes.c_float), _ptr(A_log, ctypes.c_float), _ptr(B, ctypes.c_float),
        _ptr(C, ctypes.c_float), _ptr(D, ctypes.c_float), _ptr(z, ctypes.c_float), _ptr(h0, ctypes.c_double),
        None, nrows, _ptr(y, ctypes.c_double), _ptr(mag, ctypes.c_double), _ptr(last, ctypes.c_double),
        batch, L, Dm, N)
    if st != 0:
        raise RuntimeError(f"oracle_ss_fwd_dtproj_rows failed with status {st}")
    y = y.reshape(batch, Dm, L).transpose(0, 2, 1)
    mag = mag.reshape(batch, Dm, L).transpose(0, 2, 1)
    return np.ascontiguousarray(y), last.reshape(batch, Dm, N), np.ascontiguousarray(mag)


def ss_fwd_chunked(u, delta_raw, delta_bias, A_log, B, C, D, z, chunk, h0=None):
    """fp64 chunked evaluation with the pair operator and a carry (starting from h0, or
    zeros); same returns as ss_fwd(rows=None) minus mag."""
    u = _f32(u, name="u")
    batch, L, Dm = u.shape
    A_log = _f32(A_log, name="A_log")
    N = A_log.shape[1]
    args = [u, _f32(delta_raw, (batch, L, Dm)), _f32(delta_bias, (Dm,)), A_log,
            _f32(B, (batch, L, N)), _f32(C, (batch, L, N)), _f32(D, (Dm,)), _f32(z, (batch, L, Dm))]
    y = np.empty((batch * Dm, L), np.float64)
    last = np.empty((batch * Dm, N), np.float64)
    h0 = _h0(h0, batch, Dm, N)
    st = _load().oracle_ss_fwd_chunked(*[_ptr(a, ctypes.c_float) for a in args], _ptr(h0, ctypes.c_double),
                                       _ptr(y, ctypes.c_double), _ptr(last, ctypes.c_double),
                                       batch, L, Dm, N, int(chunk))
    if st != 0:
        raise RuntimeError(f"oracle_ss_fwd_chunked failed with status {st}")
    y = np.ascontiguousarray(y.reshape(batch, Dm, L).transpose(0, 2, 1))
    return y, last.reshape(batch, Dm, N)


def ss_step(state, x, delta_raw, delta_bias, A_log, B, C, D, z):
    """One decode step in fp64.  state [batch, Dm, N] (any float dtype, not modified);
    x, delta_raw, z [batch, Dm]; B, C [batch, N].  Returns (y [batch, Dm], new_state, mag)."""
    st64 = np.array(state, dtype=np.float64, copy=True, order="C")
    batch, Dm, N = st64.shape
    x = _f32(x, (batch, Dm), "x")
    args = [x, _f32(delta_raw, (batch, Dm), "delta_raw"), _f32(delta_bias, (Dm,), "delta_bias"),
            _f32(A_log, (Dm, N), "A_log"), _f32(B, (batch, N), "B"), _f32(C, (batch, N), "C"),
            _f32(D, (Dm,), "D"), _f32(z, (batch, Dm), "z")]
    y = np.empty((batch, Dm), np.float64)
    mag = np.empty((batch, Dm), np.float64)
    st = _load().oracle_ss_step(_ptr(st64, ctypes.c_double), *[_ptr(a, ctypes.c_float) for a in args],
                                _ptr(y, ctypes.c_double), _ptr(mag, ctypes.c_double), batch, Dm, N)
    if st != 0:
        raise RuntimeError(f"oracle_ss_step failed with status {st}")
    return y, st64, mag


def conv1d(x, w, bias=None, window=None, act=True):
    """Causal depthwise conv1d in fp64.  x [batch, L, Dm] (float32 values); w [Dm, K];
    bias [Dm] or None; window [batch, Dm, K-1] (the samples before t = 0, oldest first; None:
    zeros); act: apply silu.  Returns (out [batch, L, Dm], window_out [batch, Dm, K-1])."""
    x = _f32(x, name="x")
    if x.ndim != 3:
        raise ValueError("x must be [batch, L, Dm]")
    batch, L, Dm = x.shape
    w = _f32(w, name="w")
    if w.ndim != 2 or w.shape[0] != Dm:
        raise ValueError(f"w must be [Dm, K], got {w.shape}")
    K = w.shape[1]
    bias = _f32(bias, (Dm,), "bias")
    win = None
    if window is not None:
        win = np.ascontiguousarray(np.asarray(window, dtype=np.float64))
        if win.shape != (batch, Dm, K - 1):
            raise ValueError(f"window: expected shape {(batch, Dm, K - 1)}, got {win.shape}")
    out = np.empty((batch, L, Dm), np.float64)
    wout = np.empty((batch, Dm, K - 1), np.float64)
    st = _load().oracle_conv1d(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(bias, ctypes.c_float),
                               _ptr(win, ctypes.c_double), _ptr(out, ctypes.c_double), _ptr(wout, ctypes.c_double),
                               batch, L, Dm, K, int(bool(act)))
    if st != 0:
        raise RuntimeError(f"oracle_conv1d failed with status {st}")
    return out, wout


def ss_bwd(u, delta_raw, delta_bias, A_log, B, C, D, z, dy, h0=None, dlast=None):
    """Gradients of the forward scan in fp64 for upstream gradients dy [batch, L, Dm] (of y)
    and dlast [batch, Dm, N] (of last_state, or None).  Returns a dict with du, ddelta_raw, dz
    [batch, L, Dm]; dB, dC [batch, L, N]; dA_log [Dm, N]; dD, ddelta_bias [Dm]; dh0 [batch, Dm, N]."""
    u = _f32(u, name="u")
    batch, L, Dm = u.shape
    A_log = _f32(A_log, name="A_log")
    N = A_log.shape[1]
    args = [u, _f32(delta_raw, (batch, L, Dm)), _f32(delta_bias, (Dm,)), A_log, _f32(B, (batch, L, N)),
            _f32(C, (batch, L, N)), _f32(D, (Dm,)), _f32(z, (batch, L, Dm))]
    h0 = _h0(h0, batch, Dm, N)
    dy = _f32(dy, (batch, L, Dm), "dy")
    dl = None if dlast is None else _h0(dlast, batch, Dm, N)
    out = {k: np.zeros(sh, np.float64) for k, sh in (
        ("du", (batch, L, Dm)), ("ddelta_raw", (batch, L, Dm)), ("dz", (batch, L, Dm)), ("dB", (batch, L, N)),
        ("dC", (batch, L, N)), ("dA_log", (Dm, N)), ("dD", (Dm,)), ("ddelta_bias", (Dm,)), ("dh0", (batch, Dm, N)))}
    st = _load().oracle_ss_bwd(*[_ptr(a, ctypes.c_float) for a in args], _ptr(h0, ctypes.c_double),
                               _ptr(dy, ctypes.c_float), _ptr(dl, ctypes.c_double),
                               *[_ptr(out[k], ctypes.c_double) for k in ("du", "ddelta_raw", "dz", "dB", "dC",
                                                                         "dA_log", "dD", "ddelta_bias", "dh0")],
                               batch, L, Dm, N)
    if st != 0:
        raise RuntimeError(f"oracle_ss_bwd failed with status {st}")
    return out
