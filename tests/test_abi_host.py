"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/selscan.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import selective_state_space_scan_gb300 as ss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = ss.lib()
    names = _declared_functions()
    assert {"ss_fwd", "ss_step", "ss_status_string", "ss_device_error", "ss_version"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings():
    assert ss.version() >= 100
    for code in range(5):
        assert ss.status_string(code).startswith("SS_")


def _fwd(**kw):
    args = dict(u=None, delta_raw=None, delta_bias=None, A_log=None, B=None, C=None, D=None, z=None,
                y=None, last=None, batch=1, L=8, Dm=8, N=16, strides=None)
    args.update(kw)
    lib = ss.lib()
    return lib.ss_fwd(args["u"], args["delta_raw"], args["delta_bias"], args["A_log"], args["B"],
                      args["C"], args["D"], args["z"], args["y"], args["last"], args["batch"],
                      args["L"], args["Dm"], args["N"], args["strides"], None)


FAKE = 0x10000   # never dereferenced: these calls fail validation before any device access


def test_fwd_rejects_bad_sizes_on_host():
    assert _fwd(N=0) == 2 and _fwd(N=17) == 2           # SS_ERR_UNSUPPORTED
    assert _fwd(batch=-1) == 1 and _fwd(L=-1) == 1 and _fwd(Dm=-5) == 1
    assert _fwd(batch=0) == 0 and _fwd(Dm=0) == 0         # no-ops


def test_fwd_rejects_null_and_misaligned_on_host():
    full = dict(u=FAKE, delta_raw=FAKE, A_log=FAKE, B=FAKE, C=FAKE, y=FAKE)
    assert _fwd(**{**full, "u": None}) == 1
    assert _fwd(**{**full, "A_log": None}) == 1
    assert _fwd(**{**full, "y": None}) == 1
    assert _fwd(**{**full, "u": FAKE + 2}) == 3            # fp32 pointer not 4-byte aligned
    assert _fwd(**{**full, "A_log": FAKE + 1}) == 3
    s = ss.FwdStrides(7, 64, 8, 64, 8, 0, 0, 64, 8, 128, 16, 128, 16)
    assert _fwd(**full, strides=ctypes.byref(s)) == 1     # unknown io dtype
    s = ss.FwdStrides(ss.SS_BF16, 64, 8, 64, 8, 0, 0, 64, 8, 128, 16, 128, 16)
    assert _fwd(**{**full, "u": FAKE + 1}, strides=ctypes.byref(s)) == 3
    s = ss.FwdStrides(ss.SS_F32, 64, -8, 64, 8, 0, 0, 64, 8, 128, 16, 128, 16)
    assert _fwd(**full, strides=ctypes.byref(s)) == 1     # negative stride


def test_step_rejects_bad_arguments_on_host():
    lib = ss.lib()
    call = lambda **kw: lib.ss_step(kw.get("state", FAKE), kw.get("x", FAKE), FAKE, None, FAKE,
                                    FAKE, FAKE, None, None, kw.get("y", FAKE), kw.get("batch", 2),
                                    kw.get("Dm", 8), kw.get("N", 16), None, None)
    assert call(N=0) == 2 and call(N=20) == 2
    assert call(batch=-1) == 1
    assert call(batch=0) == 0
    assert call(state=None) == 1 and call(y=None) == 1
    assert call(state=FAKE + 2) == 3


def test_conv1d_rejects_bad_arguments_on_host():
    lib = ss.lib()
    call = lambda **kw: lib.ss_conv1d(kw.get("x", FAKE), kw.get("w", FAKE), None, kw.get("out", FAKE), None, None,
                                      kw.get("batch", 2), kw.get("L", 8), kw.get("Dm", 8), 1, kw.get("strides"), None)
    assert call(batch=-1) == 1 and call(L=-1) == 1
    assert call(batch=0) == 0 and call(Dm=0) == 0
    assert call(w=None) == 1
    s = ss.ConvStrides(9, 64, 8, 64, 8)
    assert call(strides=ctypes.byref(s)) == 1              # unknown io dtype


def test_bwd_rejects_bad_arguments_on_host():
    lib = ss.lib()
    assert lib.ss_bwd_workspace_size(0, 8, 8, 16) == 0 and lib.ss_bwd_workspace_size(1, 8, 8, 17) == 0

    def call(**kw):
        p = [FAKE] * 20
        p[2] = p[6] = p[7] = p[8] = p[10] = p[13] = p[17] = p[18] = p[19] = None   # optional ones absent
        for i, v in kw.get("ptrs", {}).items():
            p[i] = v
        return lib.ss_bwd(*p, kw.get("batch", 1), kw.get("L", 8), kw.get("Dm", 8), kw.get("N", 16), None, FAKE,
                          1 << 20, None)
    assert call(N=0) == 2 and call(N=17) == 2
    assert call(batch=-1) == 1
    assert call(batch=0) == 0
    assert call(ptrs={3: None}) == 1                       # A_log
    assert call(ptrs={11: FAKE + 2}) == 3                  # du not 4-byte aligned


def test_dtproj_and_host_calls_reject_bad_arguments_on_host():
    lib = ss.lib()
    dt = lambda R, **kw: lib.ss_fwd_dtproj(FAKE, FAKE, FAKE, R, None, FAKE, FAKE, FAKE, None, None, FAKE, None, None,
                                           kw.get("batch", 1), 8, 8, 16, kw.get("strides"), None)
    assert dt(6) == 2 and dt(0) == 2 and dt(68) == 2       # rank not a multiple of 4 in 4..64
    assert dt(8, batch=-1) == 1
    s = ss.FwdStrides(ss.SS_BF16, 64, 8, 64, 8, 0, 0, 64, 8, 128, 16, 128, 16)
    assert dt(8, strides=ctypes.byref(s)) == 2              # bf16 I/O
    assert lib.ss_fwd_host_workspace_size(8, 2048, 1536, 16, ss.SS_F32) > 0
    assert lib.ss_fwd_host_workspace_size(8, 2048, 1536, 16, 5) == 0
    host = lambda **kw: lib.ss_fwd_host(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                        kw.get("batch", 1), 8, 8, kw.get("N", 16), kw.get("io", ss.SS_F32), FAKE,
                                        1 << 20, None)
    assert host(N=0) == 2 and host(io=3) == 1 and host(batch=-1) == 1
    assert host(batch=0) == 0


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


def test_outputs_whose_elements_share_words_are_rejected_on_host():
    """y (forward), y and the state (decode) and out (conv1d) are written, so no two of their
    elements may sit at one address; inputs may (a broadcast).  Rejected before any device
    access; a layout that passes reaches the device checks (SS_ERR_CUDA without a GPU)."""
    full = dict(u=FAKE, delta_raw=FAKE, A_log=FAKE, B=FAKE, C=FAKE, y=FAKE)
    # batch 2, L 8, Dm 8: (y_b, y_l)
    for y_b, y_l in ((0, 8), (32, 8), (8, 8)):               # broadcast rows, rows running into each other
        s = ss.FwdStrides(ss.SS_F32, 64, 8, 64, 8, 0, 0, y_b, y_l, 128, 16, 128, 16)
        assert _fwd(**full, batch=2, strides=ctypes.byref(s)) == 1, (y_b, y_l)
    s = ss.FwdStrides(ss.SS_F32, 0, 8, 0, 8, 0, 0, 64, 8, 0, 16, 0, 16)   # inputs broadcast over batch: allowed
    ok = [_fwd(**full, batch=2, strides=ctypes.byref(s))]
    for y_b, y_l in ((64, 8), (8, 16), (1000, 9)):           # contiguous, batch rows interleaved, padded
        s = ss.FwdStrides(ss.SS_F32, 64, 8, 64, 8, 0, 0, y_b, y_l, 128, 16, 128, 16)
        ok.append(_fwd(**full, batch=2, strides=ctypes.byref(s)))
    if _no_gpu():                                              # (with a GPU the fake pointers fail the device check)
        assert ok == [4] * len(ok), ok                         # past the layout checks, stopped at the device
    lib = ss.lib()

    def step(**kw):
        st = ss.StepStrides(ss.SS_F32, 8, 8, 0, kw.get("y_b", 8), 16, 16, kw.get("state_b", 128), kw.get("state_d", 16))
        return lib.ss_step(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE, 2, 8, 16, ctypes.byref(st), None)
    assert step(state_b=0) == 1                                # both rows on one state
    assert step(state_b=112) == 1                              # row 1 starts inside row 0
    assert step(y_b=4) == 1
    if _no_gpu():
        assert step() == 4 and step(state_b=16, state_d=32) == 4   # contiguous; rows interleaved

    def conv(out_b, out_l):
        cs = ss.ConvStrides(ss.SS_F32, 64, 8, out_b, out_l)
        return lib.ss_conv1d(FAKE, FAKE, None, FAKE, None, None, 2, 8, 8, 1, ctypes.byref(cs), None)
    assert conv(0, 8) == 1 and conv(40, 8) == 1
    if _no_gpu():
        assert conv(64, 8) == 4
