"""GB300-native Mamba selective scan: Python binding of libselscan's C ABI.

Argument marshalling only: every step of the scan runs in the CUDA library
(``include/selscan.h``).  PyTorch supplies device memory and the current stream.
There is no CPU path: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

__all__ = ["ss_fwd", "ss_fwd_ckpt", "ss_fwd_dtproj", "ss_fwd_host", "ss_step", "ss_step_layers", "ss_fwd_summary", "ss_carry_compose", "ss_conv1d", "ss_bwd", "ss_fwd_workspace_size", "SelscanError", "lib", "device_error",
           "version", "status_string", "SS_F32", "SS_BF16", "FwdStrides", "StepStrides", "ConvStrides"]

SS_F32, SS_BF16 = 0, 1
_STATUS = {0: "SS_OK", 1: "SS_ERR_INVALID_ARG", 2: "SS_ERR_UNSUPPORTED", 3: "SS_ERR_MISALIGNED",
           4: "SS_ERR_CUDA"}


class SelscanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class FwdStrides(ctypes.Structure):
    _fields_ = [("io_dtype", ctypes.c_int32)] + [(n, ctypes.c_int64) for n in (
        "u_b", "u_l", "delta_b", "delta_l", "z_b", "z_l", "y_b", "y_l", "B_b", "B_l", "C_b", "C_l")]


class ConvStrides(ctypes.Structure):
    _fields_ = [("io_dtype", ctypes.c_int32)] + [(n, ctypes.c_int64) for n in ("x_b", "x_l", "out_b", "out_l")]


class StepStrides(ctypes.Structure):
    _fields_ = [("io_dtype", ctypes.c_int32)] + [(n, ctypes.c_int64) for n in (
        "x_b", "delta_b", "z_b", "y_b", "B_b", "C_b", "state_b", "state_d")]


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libselscan (built in-tree first if missing or stale)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        L.ss_fwd.argtypes = [vp] * 10 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp]
        L.ss_fwd.restype = ctypes.c_int
        L.ss_fwd_ws.argtypes = [vp] * 10 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp, ctypes.c_size_t, vp]
        L.ss_fwd_ws.restype = ctypes.c_int
        L.ss_fwd_h0.argtypes = [vp] * 11 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp, ctypes.c_size_t, vp]
        L.ss_fwd_h0.restype = ctypes.c_int
        L.ss_fwd_dtproj.argtypes = [vp] * 3 + [i64] + [vp] * 9 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp]
        L.ss_fwd_dtproj.restype = ctypes.c_int
        L.ss_fwd_host.argtypes = [vp] * 10 + [i64] * 4 + [ctypes.c_int32, vp, ctypes.c_size_t, vp]
        L.ss_fwd_host.restype = ctypes.c_int
        L.ss_fwd_host_workspace_size.argtypes = [i64] * 4 + [ctypes.c_int32]
        L.ss_fwd_host_workspace_size.restype = ctypes.c_size_t
        L.ss_fwd_workspace_size.argtypes = [i64] * 4 + [ctypes.c_int32]
        L.ss_fwd_workspace_size.restype = ctypes.c_size_t
        L.ss_step.argtypes = [vp] * 10 + [i64] * 3 + [ctypes.POINTER(StepStrides), vp]
        L.ss_step.restype = ctypes.c_int
        L.ss_step_layers.argtypes = [ctypes.POINTER(StepLayer), i64, i64, i64, i64, ctypes.POINTER(StepStrides), vp]
        L.ss_step_layers.restype = ctypes.c_int
        L.ss_fwd_summary.argtypes = [vp] * 7 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp]
        L.ss_fwd_summary.restype = ctypes.c_int
        L.ss_carry_compose.argtypes = [vp] * 4 + [i64] * 4 + [vp]
        L.ss_carry_compose.restype = ctypes.c_int
        L.ss_conv1d.argtypes = [vp] * 6 + [i64] * 3 + [ctypes.c_int32, ctypes.POINTER(ConvStrides), vp]
        L.ss_conv1d.restype = ctypes.c_int
        L.ss_bwd.argtypes = [vp] * 20 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp, ctypes.c_size_t, vp]
        L.ss_bwd.restype = ctypes.c_int
        L.ss_bwd_workspace_size.argtypes = [i64] * 4
        L.ss_bwd_workspace_size.restype = ctypes.c_size_t
        L.ss_bwd_ckpt.argtypes = [vp] * 21 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp, ctypes.c_size_t, vp]
        L.ss_bwd_ckpt.restype = ctypes.c_int
        L.ss_fwd_ckpt.argtypes = [vp] * 12 + [i64] * 4 + [ctypes.POINTER(FwdStrides), vp, ctypes.c_size_t, vp]
        L.ss_fwd_ckpt.restype = ctypes.c_int
        L.ss_fwd_ckpt_size.argtypes = [i64] * 4
        L.ss_fwd_ckpt_size.restype = ctypes.c_size_t
        L.ss_status_string.argtypes = [ctypes.c_int]
        L.ss_status_string.restype = ctypes.c_char_p
        L.ss_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.ss_device_error.restype = ctypes.c_int
        L.ss_version.argtypes = []
        L.ss_version.restype = ctypes.c_int
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    try:
        return lib().ss_status_string(int(status)).decode()
    except OSError:
        return _STATUS.get(int(status), f"status {status}")


def version() -> int:
    return int(lib().ss_version())


def device_error(clear: bool = False) -> int:
    bits = ctypes.c_uint32(0)
    st = lib().ss_device_error(ctypes.byref(bits), int(bool(clear)))
    if st != 0:
        raise SelscanError(st, "ss_device_error")
    return int(bits.value)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _io_code(dtype) -> int:
    import torch
    if dtype == torch.float32:
        return SS_F32
    if dtype == torch.bfloat16:
        return SS_BF16
    raise TypeError(f"io tensors must be float32 or bfloat16, got {dtype}")


def _check_inner(t, name):
    if t is not None and t.dim() > 0 and t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"{name}: the last axis must have stride 1")


_WORKSPACES = {}
_WS_SIZES = {}


def workspace_for(device, stream, nbytes: int, purpose: str = "fwd"):
    """A zero-filled, 256-byte aligned device buffer of at least nbytes, cached per (device,
    stream, purpose) and grown when needed; calls on one stream are ordered, so they never
    overlap on the GPU while sharing it.  The forward schedules' hand-over flags and the
    backward's checkpoints live in separate buffers (the flags must never see checkpoint bits).
    ``stream`` is the torch stream the calls run on (None: the device's current stream).  The
    buffer is allocated and zero-filled on that stream, so the fill is ordered before its first
    use, and when a larger buffer replaces it the caching allocator hands the old memory only to
    later work on the same stream."""
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (str(device), s.cuda_stream, purpose)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(s):
            ws = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def ss_fwd_workspace_size(batch, L, Dm, N, io_dtype=SS_F32) -> int:
    """Bytes of workspace ss_fwd_ws / ss_fwd_h0 need on the current device (0: none)."""
    import torch
    key = (torch.cuda.current_device() if torch.cuda.is_available() else -1, batch, L, Dm, N, io_dtype)
    if key not in _WS_SIZES:
        _WS_SIZES[key] = int(lib().ss_fwd_workspace_size(batch, L, Dm, N, io_dtype))
    return _WS_SIZES[key]


def ss_fwd(u, delta_raw, delta_bias, A_log, B, C, D=None, z=None, y=None, last_state=None,
           stream=None, workspace=False, h0=None):
    """Selective-scan forward pass through the C ABI.

    u, delta_raw, z: [batch, L, Dm]; B, C: [batch, L, N] (same dtype, float32 or bfloat16);
    A_log [Dm, N], D and delta_bias [Dm]: float32.  ``y`` (allocated like u when None) and
    ``last_state`` ([batch, Dm, N] float32, optional) are written.  Returns y.
    h0 ([batch, Dm, N] float32, optional) is the state before step 0 (ss_fwd_h0); it may be
    last_state itself.
    workspace=False (default) calls ss_fwd: one CTA per channel tile over the whole sequence, or,
    with more tiles than the GPU holds at once, clusters of CTAs that split their tiles' work
    evenly (the cluster-balanced schedule), or for few tiles the single-launch time split.
    workspace=True passes a workspace cached per (device, stream), which enables the balanced
    schedule (equal work per CTA) or, for few channel tiles, the time-split one (ss_fwd_ws).
    """
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    io = _io_code(u.dtype)
    if y is None:
        y = torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device)
    for name, t in (("u", u), ("delta_raw", delta_raw), ("z", z), ("y", y), ("B", B), ("C", C)):
        _check_inner(t, name)
    if h0 is not None and (h0.dtype != torch.float32 or not h0.is_contiguous() or
                           tuple(h0.shape) != (batch, Dm, N)):
        raise ValueError("h0 must be a contiguous float32 [batch, Dm, N] tensor")
    s = FwdStrides(io, u.stride(0), u.stride(1), delta_raw.stride(0), delta_raw.stride(1),
                   z.stride(0) if z is not None else 0, z.stride(1) if z is not None else 0,
                   y.stride(0), y.stride(1), B.stride(0), B.stride(1), C.stride(0), C.stride(1))
    head = (_ptr(u), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(C),
            _ptr(D), _ptr(z), _ptr(y), _ptr(last_state))
    dims = (batch, L, Dm, N, ctypes.byref(s))
    nbytes = ss_fwd_workspace_size(batch, L, Dm, N, io) if workspace and batch * L * Dm > 0 else 0
    sh = _stream_handle(stream)
    ws_ptr, ws_len = None, 0
    if nbytes:
        ws = workspace_for(u.device, stream, nbytes)
        ws_ptr, ws_len = ws.data_ptr(), ws.numel()
    if h0 is not None:
        st = lib().ss_fwd_h0(*head, _ptr(h0), *dims, ws_ptr, ws_len, sh)
        where = "ss_fwd_h0"
    elif nbytes:
        st = lib().ss_fwd_ws(*head, *dims, ws_ptr, ws_len, sh)
        where = "ss_fwd_ws"
    else:
        st = lib().ss_fwd(*head, *dims, sh)
        where = "ss_fwd"
    if st != 0:
        raise SelscanError(st, where)
    return y


def ss_fwd_dtproj(u, dt_low, W_dt, delta_bias, A_log, B, C, D=None, z=None, y=None, last_state=None,
                  h0=None, stream=None):
    """Forward pass with the low-rank time-step projection folded in (ss_fwd_dtproj):
    delta_raw[b,t,d] = sum_k W_dt[d,k] dt_low[b,t,k] is computed inside the kernel.
    dt_low [batch, L, R] float32 (last axis stride 1), W_dt [Dm, R] float32 contiguous; the rest
    as ss_fwd (float32 I/O).  Returns y."""
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    R = W_dt.shape[1]
    io = _io_code(u.dtype)
    if y is None:
        y = torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device)
    for name, t in (("u", u), ("dt_low", dt_low), ("z", z), ("y", y), ("B", B), ("C", C)):
        _check_inner(t, name)
    if not W_dt.is_contiguous() or W_dt.dtype != torch.float32:
        raise ValueError("W_dt must be a contiguous float32 [Dm, R] tensor")
    s = FwdStrides(io, u.stride(0), u.stride(1), dt_low.stride(0), dt_low.stride(1),
                   z.stride(0) if z is not None else 0, z.stride(1) if z is not None else 0,
                   y.stride(0), y.stride(1), B.stride(0), B.stride(1), C.stride(0), C.stride(1))
    st = lib().ss_fwd_dtproj(_ptr(u), _ptr(dt_low), _ptr(W_dt), R, _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _ptr(y), _ptr(last_state), _ptr(h0), batch, L, Dm, N,
                             ctypes.byref(s), _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_fwd_dtproj")
    return y


def ss_fwd_host(u, delta_raw, delta_bias, A_log, B, C, D=None, z=None, y=None, last_state=None, stream=None,
                device=None):
    """Forward pass on host (CPU) tensors (ss_fwd_host): copies in, scan and copies back happen
    inside the call, overlapped over groups of batch rows.  All tensors are contiguous CPU tensors
    (pinned memory for asynchronous copies); ``y`` and ``last_state`` (optional) are written and
    valid once the stream is synchronised.  The call runs on ``device`` (default: the current one;
    ``stream`` must be on it).  The device staging workspace is cached per (device, stream).
    Returns y."""
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    io = _io_code(u.dtype)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if y is None:
        y = torch.empty((batch, L, Dm), dtype=u.dtype, pin_memory=True)
    for name, t in (("u", u), ("delta_raw", delta_raw), ("z", z), ("B", B), ("C", C), ("y", y), ("A_log", A_log),
                    ("D", D), ("delta_bias", delta_bias), ("last_state", last_state)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, the call on {dev}")
    with torch.cuda.device(dev):          # the library runs on the current device
        sh = _stream_handle(stream)
        nbytes = int(lib().ss_fwd_host_workspace_size(batch, L, Dm, N, io))
        ws = workspace_for(dev, stream, nbytes, purpose="host") if nbytes else None
        st = lib().ss_fwd_host(_ptr(u), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D),
                               _ptr(z), _ptr(y), _ptr(last_state), batch, L, Dm, N, io,
                               None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(), sh)
    if st != 0:
        raise SelscanError(st, "ss_fwd_host")
    return y


def ss_step(state, x, delta_raw, delta_bias, A_log, B, C, D=None, z=None, y=None, stream=None):
    """One decode step through the C ABI: updates ``state`` [batch, Dm, N] (float32) in place
    and returns y [batch, Dm] (allocated like x when None)."""
    import torch
    batch, Dm, N = state.shape
    io = _io_code(x.dtype)
    if y is None:
        y = torch.empty((batch, Dm), dtype=x.dtype, device=x.device)
    for name, t in (("x", x), ("delta_raw", delta_raw), ("z", z), ("y", y), ("B", B), ("C", C),
                    ("state", state)):
        _check_inner(t, name)
    s = StepStrides(io, x.stride(0), delta_raw.stride(0), z.stride(0) if z is not None else 0,
                    y.stride(0), B.stride(0), C.stride(0), state.stride(0), state.stride(1))
    st = lib().ss_step(_ptr(state), _ptr(x), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log),
                       _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(y), batch, Dm, N, ctypes.byref(s),
                       _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_step")
    return y


def ss_fwd_summary(u, delta_raw, delta_bias, A_log, B, h_end=None, dsum=None, stream=None):
    """Summary of one sequence segment through the C ABI (ss_fwd_summary): returns (h_end
    [batch, Dm, N], dsum [batch, Dm]), the state the segment leaves from a zero start and the
    sum of its Δ (float32, allocated when None)."""
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    io = _io_code(u.dtype)
    if h_end is None:
        h_end = torch.empty((batch, Dm, N), dtype=torch.float32, device=u.device)
    if dsum is None:
        dsum = torch.empty((batch, Dm), dtype=torch.float32, device=u.device)
    for name, t in (("u", u), ("delta_raw", delta_raw), ("B", B)):
        _check_inner(t, name)
    s = FwdStrides(io, u.stride(0), u.stride(1), delta_raw.stride(0), delta_raw.stride(1), 0, 0, 0, 0,
                   B.stride(0), B.stride(1), B.stride(0), B.stride(1))
    st = lib().ss_fwd_summary(_ptr(u), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(h_end),
                              _ptr(dsum), batch, L, Dm, N, ctypes.byref(s), _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_fwd_summary")
    return h_end, dsum


def ss_carry_compose(slots, dsum, A_log, h0=None, stream=None):
    """Left-to-right composition of segment summaries in place (ss_carry_compose): slots
    [nseg, batch, Dm, N] float32 holds the segments' h_end in slots 1.. on entry and each
    segment's entering state on exit; dsum [nseg - 1, batch, Dm]; h0 the state before segment 0
    (None: zeros).  Returns slots."""
    nseg, batch, Dm, N = slots.shape
    st = lib().ss_carry_compose(_ptr(slots), _ptr(dsum) if nseg > 1 else None, _ptr(h0), _ptr(A_log), nseg, batch,
                                Dm, N, _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_carry_compose")
    return slots


class StepLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("state", "x", "delta_raw", "delta_bias", "A_log", "B", "C", "D",
                                               "z", "y")]


def ss_step_layers(layers, stream=None):
    """Many layers' decode steps in one launch through the C ABI (ss_step_layers).  ``layers`` is
    a list of dicts with the tensors of one ss_step call each (keys state, x, delta_raw,
    delta_bias, A_log, B, C and optionally D, z, y); every layer has the same sizes and strides.
    Updates each state in place and returns the list of y tensors (allocated like x when a
    layer gives none)."""
    import torch
    if not layers:
        return []
    first = layers[0]
    batch, Dm, N = first["state"].shape
    io = _io_code(first["x"].dtype)
    table = (StepLayer * len(layers))()
    ys = []
    for i, L in enumerate(layers):
        y = L.get("y")
        if y is None:
            y = torch.empty((batch, Dm), dtype=L["x"].dtype, device=L["x"].device)
        ys.append(y)
        for name in ("x", "delta_raw", "z", "B", "C", "state"):
            _check_inner(L.get(name), name)
        _check_inner(y, "y")
        table[i] = StepLayer(*[_ptr(L.get(k)) for k in ("state", "x", "delta_raw", "delta_bias", "A_log", "B", "C",
                                                        "D", "z")], _ptr(y))
    x, dr, z, B, C, state = (first["x"], first["delta_raw"], first.get("z"), first["B"], first["C"],
                             first["state"])
    s = StepStrides(io, x.stride(0), dr.stride(0), z.stride(0) if z is not None else 0, ys[0].stride(0),
                    B.stride(0), C.stride(0), state.stride(0), state.stride(1))
    st = lib().ss_step_layers(table, len(layers), batch, Dm, N, ctypes.byref(s), _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_step_layers")
    return ys


def ss_conv1d(x, weight, bias=None, out=None, window_in=None, window_out=None, silu=True, stream=None):
    """Causal depthwise conv1d (kernel 4) + optional SiLU through the C ABI.

    x [batch, L, Dm] float32 or bfloat16 (channel stride 1); weight [Dm, 4] float32; bias [Dm];
    window_in / window_out [batch, Dm, 3] float32 (the samples before t = 0, oldest first; the
    same tensor updates it in place).  ``out`` is allocated like x when None.  Returns out."""
    import torch
    batch, L, Dm = x.shape
    io = _io_code(x.dtype)
    if out is None:
        out = torch.empty((batch, L, Dm), dtype=x.dtype, device=x.device)
    for name, t in (("x", x), ("out", out)):
        _check_inner(t, name)
    s = ConvStrides(io, x.stride(0), x.stride(1), out.stride(0), out.stride(1))
    st = lib().ss_conv1d(_ptr(x), _ptr(weight), _ptr(bias), _ptr(out), _ptr(window_in), _ptr(window_out),
                         batch, L, Dm, int(bool(silu)), ctypes.byref(s), _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_conv1d")
    return out


def ss_fwd_ckpt(u, delta_raw, delta_bias, A_log, B, C, D=None, z=None, y=None, last_state=None, h0=None,
                ckpt=None, stream=None, workspace=True):
    """Forward pass for training through the C ABI (ss_fwd_ckpt): y as ss_fwd, and the
    checkpoints ss_bwd(..., ckpt=...) reads instead of a first pass of its own (16 states only).
    workspace=True passes the per-(device, stream) cached workspace (the balanced schedule).
    Returns (y, ckpt); ckpt (float32, allocated when None) has ss_fwd_ckpt_size bytes."""
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    io = _io_code(u.dtype)
    if y is None:
        y = torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device)
    for name, t in (("u", u), ("delta_raw", delta_raw), ("z", z), ("y", y), ("B", B), ("C", C)):
        _check_inner(t, name)
    nbytes = int(lib().ss_fwd_ckpt_size(batch, L, Dm, N))
    if ckpt is None:
        ckpt = torch.empty((max(nbytes, 4) // 4,), dtype=torch.float32, device=u.device)
    s = FwdStrides(io, u.stride(0), u.stride(1), delta_raw.stride(0), delta_raw.stride(1),
                   z.stride(0) if z is not None else 0, z.stride(1) if z is not None else 0,
                   y.stride(0), y.stride(1), B.stride(0), B.stride(1), C.stride(0), C.stride(1))
    ws_ptr, ws_len = None, 0
    wbytes = ss_fwd_workspace_size(batch, L, Dm, N, io) if workspace and batch * L * Dm > 0 else 0
    if wbytes:
        ws = workspace_for(u.device, stream, wbytes)
        ws_ptr, ws_len = ws.data_ptr(), ws.numel()
    st = lib().ss_fwd_ckpt(_ptr(u), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D),
                           _ptr(z), _ptr(y), _ptr(last_state), _ptr(h0), _ptr(ckpt), batch, L, Dm, N, ctypes.byref(s),
                           ws_ptr, ws_len, _stream_handle(stream))
    if st != 0:
        raise SelscanError(st, "ss_fwd_ckpt")
    return y, ckpt


def ss_bwd(dy, u, delta_raw, delta_bias, A_log, B, C, D=None, z=None, h0=None, dlast=None, stream=None, ckpt=None):
    """Gradients of ss_fwd (from h0) through the C ABI.  dy [batch, L, Dm] (gradient of y, io
    dtype); dlast [batch, Dm, N] float32 (of last_state) or None.  Returns a dict: du,
    ddelta_raw, dz (None without z) [batch, L, Dm] io dtype; dB, dC [batch, L, N], dA_log [Dm, N],
    dD, ddelta_bias [Dm], dh0 [batch, Dm, N] float32.  The workspace (chunk checkpoints) comes
    from the per-(device, stream) cache.  ckpt: the checkpoints ss_fwd_ckpt wrote on the same
    inputs and h0 (ss_bwd_ckpt: no first pass), or None."""
    import torch
    batch, L, Dm = u.shape
    N = A_log.shape[1]
    io = _io_code(u.dtype)
    for name, t in (("u", u), ("delta_raw", delta_raw), ("z", z), ("B", B), ("C", C)):
        _check_inner(t, name)
    dy = dy.contiguous()
    f32 = dict(dtype=torch.float32, device=u.device)
    g = dict(du=torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device),
             ddelta_raw=torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device),
             dz=torch.empty((batch, L, Dm), dtype=u.dtype, device=u.device) if z is not None else None,
             dB=torch.empty((batch, L, N), **f32), dC=torch.empty((batch, L, N), **f32),
             dA_log=torch.empty((Dm, N), **f32), dD=torch.empty((Dm,), **f32),
             ddelta_bias=torch.empty((Dm,), **f32), dh0=torch.empty((batch, Dm, N), **f32))
    s = FwdStrides(io, u.stride(0), u.stride(1), delta_raw.stride(0), delta_raw.stride(1),
                   z.stride(0) if z is not None else 0, z.stride(1) if z is not None else 0,
                   0, 0, B.stride(0), B.stride(1), C.stride(0), C.stride(1))
    sh = _stream_handle(stream)
    nbytes = int(lib().ss_bwd_workspace_size(batch, L, Dm, N))
    ws = workspace_for(u.device, stream, nbytes, purpose="bwd") if nbytes else None
    head = (_ptr(u), _ptr(delta_raw), _ptr(delta_bias), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0))
    tail = (_ptr(dy), _ptr(dlast), _ptr(g["du"]), _ptr(g["ddelta_raw"]), _ptr(g["dz"]), _ptr(g["dB"]), _ptr(g["dC"]),
            _ptr(g["dA_log"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]), batch, L, Dm, N, ctypes.byref(s),
            None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(), sh)
    if ckpt is not None:
        st = lib().ss_bwd_ckpt(*head, _ptr(ckpt), *tail)
        where = "ss_bwd_ckpt"
    else:
        st = lib().ss_bwd(*head, *tail)
        where = "ss_bwd"
    if st != 0:
        raise SelscanError(st, where)
    return g
