"""Benchmark: selective-scan forward (or decode) throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole hot path over one batch of synthetic input:
  forward workloads: one ss_fwd over the whole [batch, L, Dm] problem (softplus, the scan,
                     D skip, z gate and last_state, all in one kernel launch);
  decode workload:   the decode update of 48 layers' distinct states: one ss_step_layers launch
                     (or, with --decode-per-layer, 48 ss_step launches), replayed as a CUDA graph.
Prints one JSON line.  Inputs live in HBM before the timed region; every workload's working
set is larger than the 129 MB L2, so no flush is needed between steps.  Under torchrun each
rank runs its own copy of the workload (independent problems, no collective): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan state-updates/s (B·L·D·N) & HBM GB/s vs roofline, 1×GB300"
UNIT = "state-updates/s"
DECODE_LAYERS = 48


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mamba2p8b_bf16",
                    choices=["mamba130m", "long32k", "mamba2p8b_bf16", "decode1p4b", "tiny", "conv1d_130m",
                             "bwd_130m", "bwd_long32k", "lti_130m", "dtproj_130m"],
                    help="conv1d_130m times the causal conv1d + SiLU on the 130m layer's conv input "
                         "(its own metric, outputs/s); bwd_130m / bwd_long32k the backward scan of the 130m / "
                         "long-sequence layer; "
                         "lti_130m the forward with B and C constant over the steps; dtproj_130m the forward "
                         "with the rank-48 time-step projection folded in")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--probe", action="store_true",
                    help="print the measured results per clock per SM of ex2, rcp, lg2, tanh, FFMA and FFMA2 "
                         "(the library's pipe probe) and exit")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bwd-ckpt", action="store_true",
                    help="backward workloads: time ss_bwd with its own first pass instead of reading the "
                         "forward's checkpoints (ss_fwd_ckpt + ss_bwd_ckpt)")
    ap.add_argument("--variant", default=None,
                    help="pin the forward kernel as family,q,tma (family 0 channel-lane / 1 segment-lane; "
                         "q warps per CTA 1|2|4 or 0 auto; tma 1|0|-1 auto); default: the library's choice")
    ap.add_argument("--workspace", action="store_true", default=True,
                    help="(default) call the forward pass with the binding's cached workspace (ss_fwd_ws: the "
                         "balanced or the time-split schedule)")
    ap.add_argument("--decode-per-layer", action="store_true",
                    help="decode workload: time 48 ss_step launches (one per layer) instead of one "
                         "ss_step_layers launch over all 48")
    ap.add_argument("--no-workspace", dest="workspace", action="store_false",
                    help="call the plain ss_fwd instead (one CTA per channel tile, no workspace)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def alg_bytes(w) -> int:
    """Bytes the method must move: read u, delta_raw, z and write y ([B,L,Dm] io dtype); read
    B, C ([B,L,N]); params A_log [Dm,N], D, bias [Dm] fp32; write last_state [B,Dm,N] fp32."""
    s = w.io_bytes()
    if w.name.startswith("decode"):
        # per layer: x, delta_raw, z read + y write [B,Dm]; B, C [B,N]; A_log, D; state r+w
        per = (4 * w.batch * w.Dm + 2 * w.batch * w.N) * s + (w.Dm * w.N + w.Dm) * 4 \
            + 2 * w.batch * w.Dm * w.N * 4
        return per * DECODE_LAYERS
    return w.batch * w.L * (4 * w.Dm + 2 * w.N) * s + w.Dm * (w.N + 2) * 4 + w.batch * w.Dm * w.N * 4


PROBE_KINDS = {"ex2": 0, "rcp": 1, "lg2": 2, "tanh": 3, "ffma": 4, "ffma2": 5}


def max_sm_mhz(clocks=None) -> tuple:
    """The SM clock the arithmetic peaks are quoted at: nvidia-smi's clocks.max.sm sampled during
    the run, else the one MEASURED_PEAKS.json recorded."""
    if clocks and clocks.get("sm_max_mhz"):
        return float(clocks["sm_max_mhz"]), "nvidia-smi clocks.max.sm"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("sm_max_mhz"):
            return float(d["sm_max_mhz"]), "MEASURED_PEAKS.json sm_max_mhz"
    raise RuntimeError("no SM clock: nvidia-smi gave none and MEASURED_PEAKS.json is absent")


class PipePeaks:
    """Arithmetic peaks of this GPU: the library's pipe probe (ss__pipe_probe: one CTA per SM,
    independent chains, SM cycle counter) gives results per clock per SM for ex2, rcp, lg2 and
    fp32 FMA;
    the SM count comes from the device properties and the clock from max_sm_mhz()."""

    def __init__(self, ss, torch, dev):
        import ctypes
        fn = ss.lib().ss__pipe_probe
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.per_clk = {}
        for name in ("ex2", "rcp", "lg2", "ffma"):
            r = ctypes.c_double(0.0)
            if fn(PROBE_KINDS[name], 4096, ctypes.byref(r)) != 0:
                raise RuntimeError(f"pipe probe {name} failed")
            self.per_clk[name] = r.value

    def ex2_per_s(self, clocks=None) -> float:
        return self.per_s("ex2", clocks)

    def per_s(self, op: str, clocks=None) -> float:
        return self.sms * self.per_clk[op] * max_sm_mhz(clocks)[0] * 1e6

    def ffma_per_s(self, clocks=None) -> float:
        return self.sms * self.per_clk["ffma"] * max_sm_mhz(clocks)[0] * 1e6

    def source(self, clocks=None) -> str:
        mhz, src = max_sm_mhz(clocks)
        return (f"{self.sms} SMs (device properties) x {self.per_clk['ex2']:.2f} ex2/clk/SM (ss__pipe_probe, "
                f"measured in this run) x {mhz:.0f} MHz ({src})")


def run_probe(args, local_rank):
    """--probe: results per clock per SM of every probed pipe operation, one JSON line."""
    import ctypes
    import torch
    import selective_state_space_scan_gb300 as ss
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    fn = ss.lib().ss__pipe_probe
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    rates = {}
    for name, kind in PROBE_KINDS.items():
        r = ctypes.c_double(0.0)
        if fn(kind, 4096, ctypes.byref(r)) != 0:
            raise RuntimeError(f"pipe probe {name} failed")
        rates[name] = round(r.value, 3)
    props = torch.cuda.get_device_properties(dev)
    print(json.dumps({"probe": "pipe results per clock per SM (ffma2: fp32 FMAs)", "per_clk_per_sm": rates,
                      "sms": props.multi_processor_count, "gpu": props.name}))
    return 0


def decay_ex2_per_step(w) -> int:
    """One exp2 per state update: the decay exp(Δ·A) of every (b, t, d, n)."""
    return updates_per_step(w)


def transcendentals_per_step(w) -> dict:
    """The method's full count of transcendentals: per (b, t, d) the N decays, softplus as
    exp and log (log1p(e^x)) and the gate's sigmoid as exp and reciprocal, i.e.
    B·L·Dm·(N+2) exp2, B·L·Dm log2 and B·L·Dm reciprocals."""
    rows = updates_per_step(w) // w.N
    return {"ex2": rows * (w.N + 2), "lg2": rows, "rcp": rows}


# Sources each timed kernel's code and launch configuration come from: a traffic figure
# measured on other sources is stale.
_COMMON_SOURCES = ("device_common.cuh", "fwd_params.h", "internal.h", "fwd_configs.h", "selscan_api.cu")
KERNEL_SOURCES = {
    "ss_fwd_lane_kernel": _COMMON_SOURCES + ("ss_fwd_lane.cuh", "fwd_lane_impl.cuh", "fwd_launch_common.cuh",
                                             "fwd_lane_f32.cu", "fwd_lane_bf16.cu", "fwd_lane_bf16w.cu",
                                             "ss_fwd_widen.cu", "ss_fwd_carry.cu", "fwd_lane_dtp.cu"),
    "ss_fwd_seg_kernel": _COMMON_SOURCES + ("ss_fwd_seg.cuh", "fwd_seg.cu", "fwd_launch_common.cuh"),
    "ss_step_kernel": _COMMON_SOURCES + ("ss_step.cu",),
    "ss_step_layers_kernel": _COMMON_SOURCES + ("ss_step.cu",),
    "ss_step_layers_staged_kernel": _COMMON_SOURCES + ("ss_step.cu",),
    "ss_conv1d_kernel": ("device_common.cuh", "host_util.h", "ss_conv1d.cu"),
    "ss_bwd_kernel": ("device_common.cuh", "host_util.h", "ss_bwd.cu"),
}


def kernel_source_hash(kernel: str = "") -> str:
    """Hash of the CUDA sources a kernel is built and launched from (all of csrc for "")."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_scan_gb300", "csrc")
    base = kernel.split("(")[0]
    if base in KERNEL_SOURCES:
        files = [os.path.join(csrc, f) for f in KERNEL_SOURCES[base]]
    else:
        files = glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) + \
            glob.glob(os.path.join(csrc, "*.h"))
    for f in sorted(set(files)):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    # one record per workload, plus "workload:kernel" for another call of the same workload
    for key in (workload, f"{workload}:{kernel}"):
        rec = tab.get(key)
        if rec and rec.get("kernel") == kernel and rec.get("source_hash") == kernel_source_hash(kernel):
            return rec.get("dram_bytes_per_launch")
    return None


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest value over all ranks (the timed region of the slowest rank)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, total_ms: float, steps: int) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time per step."""
    return units_per_rank * world / (total_ms / 1e3 / steps)


def updates_per_step(w) -> int:
    if w.name.startswith("decode"):
        return w.batch * w.Dm * w.N * DECODE_LAYERS
    return w.state_updates


def warm_up(step, args, torch, min_seconds=0.5):
    """At least W (>= 3) untimed steps, continued until the GPU has run them for min_seconds, so
    that the clock sampler (every 100 ms) sees the GPU under this load right up to the timed
    region, which follows without a gap."""
    n, t0 = 0, time.perf_counter()
    while n < max(args.warmup, 3) or time.perf_counter() - t0 < min_seconds:
        step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    return n


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.warmup_steps = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [v for v in sm if mx and v >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "warmup_steps_run": self.warmup_steps}


# ---------------------------------------------------------------------------- our arm

def make_fwd_call(w, torch, ss, dev, workspace=False):
    a = w.arrays
    io = w.io

    def up(x):
        if x is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
        return t.to(torch.bfloat16) if io == "bf16" else t

    def upf(x):
        return None if x is None else torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)

    t = dict(u=up(a["u"]), delta_raw=up(a["delta_raw"]), z=up(a["z"]), B=up(a["B"]), C=up(a["C"]),
             A_log=upf(a["A_log"]), D=upf(a["D"]), delta_bias=upf(a["delta_bias"]))
    y = torch.empty_like(t["u"])
    last = torch.empty((w.batch, w.Dm, w.N), device=dev)

    def step():
        ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                  y=y, last_state=last, workspace=workspace)
    return step, t, y, last


def make_decode_call(w0, torch, ss, dev, per_layer=False):
    from selective_state_space_scan_gb300 import synth
    layers = []
    for layer in range(DECODE_LAYERS):
        w = synth.step_inputs(w0.batch, w0.Dm, w0.N, io=w0.io, seed=w0.seed, layer=layer)
        a = w.arrays
        layers.append({k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in a.items()})
    ys = [torch.empty((w0.batch, w0.Dm), device=dev) for _ in layers]

    def eager():
        if per_layer:
            for L, y in zip(layers, ys):
                ss.ss_step(L["state"], L["x"], L["delta_raw"], L["delta_bias"], L["A_log"], L["B"], L["C"],
                           L["D"], L["z"], y=y)
        else:
            ss.ss_step_layers([dict(L, y=y) for L, y in zip(layers, ys)])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        eager()                      # warm the library on this stream before capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        eager()

    def step():
        g.replay()
    return step, layers, ys


def run_ours(args, w, rank, world, local_rank):
    import ctypes
    import torch
    import selective_state_space_scan_gb300 as ss
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks_live = PipePeaks(ss, torch, dev)
    if args.variant:
        fam, q, tma = (int(x) for x in args.variant.split(","))
        hook = ss.lib().ss__force_fwd_variant
        hook.argtypes = [ctypes.c_int] * 3
        if hook(fam, q, tma) != 0:
            raise ValueError(f"bad --variant {args.variant}")
    decode = w.name.startswith("decode")
    if decode:
        step, tensors, outs = make_decode_call(w, torch, ss, dev, per_layer=args.decode_per_layer)
    else:
        step, tensors, y, last = make_fwd_call(w, torch, ss, dev, workspace=args.workspace)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        # warm-up right before the timed region (no idle gap for the clocks to drop in)
        clk.warmup_steps = warm_up(step, args, torch)
        barrier()
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        end.record(stream)
        barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    err = ss.device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")
    if decode:
        # the library reports which decode kernel the last call launched: the staged one wherever
        # the buffers allow it (per layer too, as a table of one layer), else the per-block ones
        staged = ss.lib().ss__last_step_path() == 1
        kernel = ("ss_step_layers_staged_kernel" if staged else
                  "ss_step_kernel" if args.decode_per_layer else "ss_step_layers_kernel")
        launches = DECODE_LAYERS if args.decode_per_layer else 1
    else:
        plan = ss.lib().ss__fwd_plan
        plan.restype = ctypes.c_int
        plan.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int32, ctypes.c_int, ctypes.c_char_p, ctypes.c_int]
        buf = ctypes.create_string_buffer(128)
        launches = plan(w.batch, w.L, w.Dm, w.N, ss.SS_BF16 if w.io == "bf16" else ss.SS_F32,
                        1 if args.workspace else 0, buf, 128)
        kernel = buf.value.decode()

    # end-to-end through the public API: pinned host inputs -> device -> ss_fwd -> host output
    e2e = None
    if not args.no_e2e and not decode:
        e2e = run_e2e(args, w, torch, ss, dev, tensors, y, last, barrier)
    return dict(total_ms=total_ms, per_launch_ms=per_launch_ms, clocks=clk.summary(), e2e=e2e,
                kernel=kernel, launches=launches, peaks=peaks_live)


def run_e2e(args, w, torch, ss, dev, t, y, last, barrier):
    """The same metric through ss_fwd_host: pinned host inputs in, y and last_state back in
    pinned host memory, every copy inside the timed region (overlapped with the scan over groups
    of batch rows by the call itself)."""
    keys = [k for k in ("u", "delta_raw", "z", "B", "C", "A_log", "D", "delta_bias") if t[k] is not None]
    host = {k: t[k].cpu().pin_memory() for k in keys}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    last_host = torch.empty(last.shape, dtype=last.dtype).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = y_host.numel() * y_host.element_size() + last_host.numel() * last_host.element_size()
    stream = torch.cuda.current_stream()

    def step():
        ss.ss_fwd_host(host["u"], host["delta_raw"], host.get("delta_bias"), host["A_log"], host["B"], host["C"],
                       host.get("D"), host.get("z"), y=y_host, last_state=last_host)

    steps = max(3, min(args.steps, 10))
    for _ in range(3):
        step()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    barrier()
    ms = a.elapsed_time(b) / steps
    return dict(ms=ms, h2d=h2d, d2h=d2h)


# ---------------------------------------------------------------------------- oracle arm

def oracle_time(w, min_seconds=10.0, max_passes=50):
    """Time the fp64 oracle on the workload's full set of rows, repeated until min_seconds."""
    import oracle
    a = w.arrays
    passes, elapsed = 0, 0.0
    while passes < 1 or (elapsed < min_seconds and passes < max_passes):
        t0 = time.perf_counter()
        if w.name.startswith("decode"):
            oracle.ss_step(a["state"], a["x"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"],
                           a["C"], a["D"], a["z"])
        else:
            oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                          a["z"])
        elapsed += time.perf_counter() - t0
        passes += 1
    units = (w.batch * w.Dm * w.N if w.name.startswith("decode") else w.state_updates) * passes
    return units / elapsed, passes, elapsed, oracle.num_threads()


def oracle_sample_baseline(fn, units_per_pass, unit, sample, min_seconds=10.0, max_passes=50):
    """The oracle timed on a bounded sample of a workload: fn() is one pass over the sample,
    repeated until min_seconds; returns the cpu_baseline object."""
    import oracle
    passes, elapsed = 0, 0.0
    while passes < 1 or (elapsed < min_seconds and passes < max_passes):
        t0 = time.perf_counter()
        fn()
        elapsed += time.perf_counter() - t0
        passes += 1
    return {"value": units_per_pass * passes / elapsed, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{passes} pass(es) of {sample}, {elapsed:.1f} s of fp64 oracle time"}


def workload_config(w, extra=None, variant=None, decode_per_layer=False, call=None):
    c = {"workload": f"{w.name}: batch={w.batch} L={w.L} Dm={w.Dm} N={w.N} io={w.io}",
         "batch": w.batch, "L": w.L, "Dm": w.Dm, "N": w.N, "io": w.io, "seed": w.seed,
         "l2": "no flush: working set {:.0f} MB > 129 MB L2".format(alg_bytes(w) / 1e6)}
    if w.name.startswith("decode"):
        c["layers"] = DECODE_LAYERS
        c["graph"] = ("48 ss_step launches" if decode_per_layer else "one ss_step_layers launch over "
                      "the 48 layers") + " captured in one CUDA graph per step"
    if variant:
        c["kernel_variant"] = variant
    if call:
        c["call"] = call
    if extra:
        c.update(extra)
    return c


def time_step_fn(step, args, local_rank):
    """W warm-up calls of `step`, then K timed ones bracketed by CUDA events on the current
    stream, clocks sampled throughout.  Returns (total ms, mean per-call ms, clock summary)."""
    import torch
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        clk.warmup_steps = warm_up(step, args, torch)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end), statistics.mean(a.elapsed_time(b) for a, b in ev), clk.summary()


def bench_lti(args, local_rank):
    """ss_fwd on the 130m-shaped layer (batch 8, L 2048, Dm 1536, N 16, fp32) with B and C
    constant over the steps of each batch row (step stride 0, the LTI case): the kernel holds
    them in registers.  One launch per step."""
    import torch
    import selective_state_space_scan_gb300 as ss
    from selective_state_space_scan_gb300 import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk = PipePeaks(ss, torch, dev)
    w = synth.config("mamba130m")
    a = w.arrays
    t = {k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in a.items()}
    Bm = t["B"][:, :1].expand(-1, w.L, -1)
    Cm = t["C"][:, :1].expand(-1, w.L, -1)
    y = torch.empty_like(t["u"])
    last = torch.empty((w.batch, w.Dm, w.N), device=dev)

    def step():
        ss.ss_fwd(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], Bm, Cm, t["D"], t["z"], y=y, last_state=last)
    total_ms, launch_ms, clocks = time_step_fn(step, args, local_rank)
    err = ss.device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")
    units = updates_per_step(w)
    # read u, delta_raw, z and write y; one B and C row per batch row; params; last_state
    alg = w.batch * w.L * 4 * w.Dm * 4 + 2 * w.batch * w.N * 4 + w.Dm * (w.N + 2) * 4 + w.batch * w.Dm * w.N * 4
    hbm_peak, peak_kind = peaks()
    sfu_peak = pk.ex2_per_s(clocks)
    achieved = alg / (launch_ms / 1e3) / 1e9
    kernel = "ss_fwd_lane_kernel(lpc=4,lti)"
    out = {
        "metric": "selective-scan state-updates/s (B·L·D·N), time-invariant B/C, 1×GB300",
        "value": units * args.steps / (total_ms / 1e3), "unit": "state-updates/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "lti_130m: batch=8 L=2048 Dm=1536 N=16 io=f32, B and C at step stride 0",
                   "l2": "no flush: working set 403 MB > 129 MB L2"},
        "gpu_launches": args.steps, "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": measured_traffic("lti_130m", kernel), "kernel": kernel, "launch_ms": launch_ms,
                     "alg_bytes_per_launch": alg, "t_hbm_us": alg / (hbm_peak * 1e9) * 1e6,
                     "t_sfu_us": units / sfu_peak * 1e6}}
    if not args.no_cpu_baseline:
        import oracle
        rows = np.arange(w.Dm)                       # batch row 0, every channel
        Bl = np.broadcast_to(a["B"][:, :1], a["B"].shape).copy()
        Cl = np.broadcast_to(a["C"][:, :1], a["C"].shape).copy()
        out["cpu_baseline"] = oracle_sample_baseline(
            lambda: oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], Bl, Cl, a["D"], a["z"],
                                  rows=rows),
            w.Dm * w.L * w.N, "state-updates/s", "batch row 0 of the lti_130m workload (all channels)")
    print(json.dumps(out))
    return 0


def bench_dtproj(args, local_rank):
    """ss_fwd_dtproj on the 130m-shaped layer (batch 8, L 2048, Dm 1536, N 16, fp32) with the
    time-step projection of rank 48 (Mamba-130m's dt_rank, ceil(768 / 16)) folded in: the kernel
    reads dt_low [8, 2048, 48] and W_dt [1536, 48] instead of delta_raw.  One launch per step."""
    import torch
    import selective_state_space_scan_gb300 as ss
    from selective_state_space_scan_gb300 import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk = PipePeaks(ss, torch, dev)
    w = synth.config("mamba130m")
    a = w.arrays
    R = 48
    g = synth.rng_for(1, 13)
    t = {k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in a.items()}
    dt_low = torch.from_numpy((0.5 * g.standard_normal((w.batch, w.L, R))).astype(np.float32)).to(dev)
    W_dt = torch.from_numpy((g.standard_normal((w.Dm, R)) / np.sqrt(R)).astype(np.float32)).to(dev)
    y = torch.empty_like(t["u"])
    last = torch.empty((w.batch, w.Dm, w.N), device=dev)

    def step():
        ss.ss_fwd_dtproj(t["u"], dt_low, W_dt, t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"], y=y,
                         last_state=last)
    total_ms, launch_ms, clocks = time_step_fn(step, args, local_rank)
    err = ss.device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")
    units = updates_per_step(w)
    # read u, z and write y; dt_low; B, C; params (W_dt, A_log, D, bias); last_state
    alg = (w.batch * w.L * (3 * w.Dm + R + 2 * w.N) * 4 + w.Dm * (R + w.N + 2) * 4 + w.batch * w.Dm * w.N * 4)
    hbm_peak, peak_kind = peaks()
    sfu_peak = pk.ex2_per_s(clocks)
    fma_peak = pk.ffma_per_s(clocks)                               # fp32 FMAs per second
    achieved = alg / (launch_ms / 1e3) / 1e9
    kernel = "ss_fwd_lane_kernel(lpc=4,dtproj)"
    out = {
        "metric": "selective-scan state-updates/s (B·L·D·N), dt_proj folded in, 1×GB300",
        "value": units * args.steps / (total_ms / 1e3), "unit": "state-updates/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "dtproj_130m: batch=8 L=2048 Dm=1536 N=16 dt_rank=48 io=f32",
                   "l2": "no flush: working set 310 MB > 129 MB L2"},
        "gpu_launches": args.steps, "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": measured_traffic("dtproj_130m", kernel), "kernel": kernel, "launch_ms": launch_ms,
                     "alg_bytes_per_launch": alg, "t_hbm_us": alg / (hbm_peak * 1e9) * 1e6,
                     "t_sfu_us": units / sfu_peak * 1e6,
                     "t_fma_us": w.batch * w.L * w.Dm * R / fma_peak * 1e6}}
    if not args.no_cpu_baseline:
        import oracle
        dl, Wn = dt_low[:1].cpu().numpy(), W_dt.cpu().numpy()
        one = {k: (None if v is None else (v[:1] if v.ndim == 3 else v)) for k, v in a.items()}
        out["cpu_baseline"] = oracle_sample_baseline(
            lambda: oracle.ss_fwd_dtproj(one["u"], dl, Wn, one["delta_bias"], one["A_log"], one["B"], one["C"],
                                         one["D"], one["z"]),
            w.Dm * w.L * w.N, "state-updates/s", "batch row 0 of the dtproj_130m workload (all channels)")
    print(json.dumps(out))
    return 0


def bench_conv1d(args, local_rank):
    """The causal conv1d + SiLU (ss_conv1d) on the conv input of the 130m-shaped layer (batch 8,
    L 2048, Dm 1536, fp32), window in and out: one launch per step."""
    import torch
    import selective_state_space_scan_gb300 as ss
    from selective_state_space_scan_gb300 import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    batch, L, Dm = 8, 2048, 1536
    g = synth.rng_for(1, 9)
    x = torch.from_numpy(g.standard_normal((batch, L, Dm), dtype=np.float32)).to(dev)
    wgt = torch.from_numpy((0.5 * g.standard_normal((Dm, 4), dtype=np.float32)).astype(np.float32)).to(dev)
    bias = torch.from_numpy((0.1 * g.standard_normal(Dm, dtype=np.float32)).astype(np.float32)).to(dev)
    win = torch.zeros((batch, Dm, 3), device=dev)
    out = torch.empty_like(x)

    def step():
        ss.ss_conv1d(x, wgt, bias, out=out, window_in=win, window_out=win, silu=True)
    total_ms, launch_ms, clocks = time_step_fn(step, args, local_rank)
    units = batch * L * Dm
    alg = 2 * units * 4 + Dm * 5 * 4 + 2 * batch * Dm * 3 * 4
    hbm_peak, peak_kind = peaks()
    achieved = alg / (launch_ms / 1e3) / 1e9
    out = {
        "metric": "causal conv1d + SiLU outputs/s (B·L·D), 1×GB300", "value": units * args.steps / (total_ms / 1e3),
        "unit": "outputs/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "conv1d_130m: batch=8 L=2048 Dm=1536 kernel=4 io=f32 silu window",
                   "l2": "no flush: working set 201 MB > 129 MB L2"},
        "gpu_launches": args.steps, "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": measured_traffic("conv1d_130m", "ss_conv1d_kernel"), "kernel": "ss_conv1d_kernel",
                     "launch_ms": launch_ms,
                     "alg_bytes_per_launch": alg}}
    if not args.no_cpu_baseline:
        import oracle
        xn, wn, bn = x.cpu().numpy(), wgt.cpu().numpy(), bias.cpu().numpy()
        out["cpu_baseline"] = oracle_sample_baseline(
            lambda: oracle.conv1d(xn, wn, bn, window=np.zeros((batch, Dm, 3)), act=True),
            units, "outputs/s", "the whole conv1d_130m workload")
    print(json.dumps(out))
    return 0


def bench_bwd(args, local_rank):
    """The backward scan (ss_bwd): gradients of every input for a random dy, on the 130m-shaped
    layer (bwd_130m: batch 8, L 2048, Dm 1536, N 16, fp32; one launch per step) or the
    long-sequence one (bwd_long32k: batch 1, L 32768; the time split, four launches per step)."""
    import torch
    import selective_state_space_scan_gb300 as ss
    from selective_state_space_scan_gb300 import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk = PipePeaks(ss, torch, dev)
    split = args.workload == "bwd_long32k"      # 48 channel tiles: the automatic time split
    w = synth.config("long32k" if split else "mamba130m")
    a = w.arrays
    t = {k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in a.items()}
    dy = torch.from_numpy(synth.rng_for(1, 12).standard_normal((w.batch, w.L, w.Dm), dtype=np.float32)).to(dev)

    # the training flow: the forward pass (ss_fwd_ckpt, outside the timed region) leaves the state
    # at every 16th step, and the backward reads them instead of refolding the sequence first
    # (ss_bwd_ckpt; the long row's time split also takes its segments' entering states from them)
    ckpt = None
    if not args.no_bwd_ckpt and w.N == 16:
        _, ckpt = ss.ss_fwd_ckpt(t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"])
        torch.cuda.synchronize()

    def step():
        ss.ss_bwd(dy, t["u"], t["delta_raw"], t["delta_bias"], t["A_log"], t["B"], t["C"], t["D"], t["z"], ckpt=ckpt)
    total_ms, launch_ms, clocks = time_step_fn(step, args, local_rank)
    units = updates_per_step(w)
    s = w.io_bytes()
    # must move: read u, delta_raw, z, dy and B, C; write du, ddelta_raw, dz and dB, dC; params
    alg = w.batch * w.L * (7 * w.Dm * s + 4 * w.N * 4) + w.Dm * (w.N + 2) * 4 * 2
    hbm_peak, peak_kind = peaks()
    achieved = alg / (launch_ms / 1e3) / 1e9
    # the SFU floor: two exp2 per state update (the forward recurrence and the adjoint one) at
    # the ex2 rate; below the HBM floor, so the bound is HBM
    sfu_peak = pk.ex2_per_s(clocks)
    t_hbm, t_sfu = alg / (hbm_peak * 1e9), 2 * units / sfu_peak
    out = {
        "metric": "selective-scan backward state-updates/s (B·L·D·N), 1×GB300",
        "value": units * args.steps / (total_ms / 1e3), "unit": "state-updates/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: batch={w.batch} L={w.L} Dm={w.Dm} N={w.N} io=f32, "
                               "all input gradients" + (", time split" if split else ""),
                   "l2": "no flush: working set > 129 MB L2",
                   "call": ("ss_bwd (its own first pass)" if ckpt is None else
                            "ss_bwd_ckpt: with the checkpoints ss_fwd_ckpt wrote (outside the timed region)" +
                            ("; the time split's local launch sweeps only the adjoint" if split else ""))},
        "gpu_launches": args.steps * ((3 if ckpt is not None else 4) if split else 1), "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": measured_traffic(args.workload, "ss_bwd_kernel"), "kernel": "ss_bwd_kernel",
                     "launch_ms": launch_ms, "launch_ms_is": "per step" if split else "per launch",
                     "t_hbm_us": t_hbm * 1e6, "t_sfu_us": t_sfu * 1e6, "alg_bytes_per_launch": alg}}
    if not args.no_cpu_baseline:
        import oracle
        one = {k: (None if v is None else (v[:1] if v.ndim == 3 else v)) for k, v in a.items()}
        dyn = dy[:1].cpu().numpy()
        if split:                                    # a 64-channel slice of the long row
            one = {k: (None if v is None else (v[..., :64] if v.ndim == 3 and v.shape[-1] == w.Dm else
                                               v[:64] if v.shape[0] == w.Dm else v)) for k, v in one.items()}
            dyn = dyn[..., :64]
        nch = dyn.shape[-1]
        out["cpu_baseline"] = oracle_sample_baseline(
            lambda: oracle.ss_bwd(one["u"], one["delta_raw"], one["delta_bias"], one["A_log"], one["B"], one["C"],
                                  one["D"], one["z"], dyn),
            nch * w.L * w.N, "state-updates/s",
            f"batch row 0 of the {args.workload} workload ({nch} channels)", min_seconds=5.0)
    print(json.dumps(out))
    return 0


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    from selective_state_space_scan_gb300 import synth
    if args.probe:
        return run_probe(args, local_rank) if rank == 0 else 0
    if args.workload in ("conv1d_130m", "bwd_130m", "bwd_long32k", "lti_130m", "dtproj_130m"):
        if args.impl == "reference" or world > 1:
            if rank == 0:
                print(json.dumps({"impl": args.impl,
                                  "unavailable": f"{args.workload} is measured on one GPU, ours only"}))
            return 0
        fn = {"conv1d_130m": bench_conv1d, "bwd_130m": bench_bwd, "bwd_long32k": bench_bwd, "lti_130m": bench_lti,
              "dtproj_130m": bench_dtproj}[args.workload]
        return fn(args, local_rank)
    w = synth.config(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return 0
        rates = []
        for _ in range(args.warmup):
            oracle_time(w, min_seconds=0.0, max_passes=1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            rate, _, _, cores = oracle_time(w, min_seconds=0.0, max_passes=1)
            rates.append(rate)
        total = time.perf_counter() - t0
        value = updates_per_step(w) * args.steps / total if not w.name.startswith("decode") \
            else w.batch * w.Dm * w.N * args.steps / total
        sample = f"one full pass of the {w.name} workload per step (fp64 oracle, OpenMP over rows)"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "io_dtype": w.io,
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res = run_ours(args, w, rank, world, local_rank)
    units = updates_per_step(w)
    ms_step = res["total_ms"] / args.steps
    value = job_throughput(units, world, res["total_ms"], args.steps)
    launch_ms = statistics.mean(res["per_launch_ms"])
    # decode: the step is per_step_launches equal launches (one per layer, or one for all layers);
    # forward: the step's launches run the scan once (time split: three passes; bf16 with a
    # workspace: the B/C widening first), so the whole step is timed as the scan's launch
    per_step_launches = res["launches"] if w.name.startswith("decode") else 1
    launch_ms = launch_ms / per_step_launches
    bytes_launch = alg_bytes(w) / per_step_launches if w.name.startswith("decode") else alg_bytes(w)
    hbm_peak, peak_kind = peaks()
    # Roofline of the dominant kernel: the slower of moving the algorithmic bytes at the
    # measured HBM copy bandwidth and issuing one exp2 per state update at the SFU rate.
    sfu_peak = res["peaks"].ex2_per_s(res["clocks"])     # ex2 / s
    ex2_launch = decay_ex2_per_step(w) / (per_step_launches if w.name.startswith("decode") else 1)
    t_hbm = bytes_launch / (hbm_peak * 1e9)
    t_sfu = ex2_launch / sfu_peak
    if t_hbm >= t_sfu:
        achieved = bytes_launch / (launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"}
    else:
        achieved = ex2_launch / (launch_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": sfu_peak / 1e12, "unit": "Tex2/s",
                "frac": achieved * 1e12 / sfu_peak,
                "peak_source": res["peaks"].source(res["clocks"])}
    if not w.name.startswith("decode") and res["launches"] > 1:
        roof["launch_ms_is"] = ("per step: " + str(res["launches"]) + " launches (the time split's passes and/or "
                                "the widening of bf16 B and C to fp32, about 1 us, before the scan)")
    per = per_step_launches if w.name.startswith("decode") else 1
    tr = {k: v / per for k, v in transcendentals_per_step(w).items()}
    # every transcendental at the probe's measured rate of its own operation (rcp and lg2 run at
    # half the ex2 rate): the SFU time of the whole op mix, against t_sfu's decays alone
    t_sfu_all = sum(tr[k] / res["peaks"].per_s(k, res["clocks"]) for k in tr)
    roof.update({"transcendentals_per_launch": tr, "t_sfu_all_us": t_sfu_all * 1e6})
    roof.update({"traffic": measured_traffic(w.name, res["kernel"]), "kernel": res["kernel"],
                 "launch_ms": launch_ms, "alg_bytes_per_launch": bytes_launch,
                 "decay_ex2_per_launch": ex2_launch, "t_hbm_us": t_hbm * 1e6, "t_sfu_us": t_sfu * 1e6})
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": w.io, "data": "synthetic",
        "config": workload_config(
            w, variant=args.variant, decode_per_layer=args.decode_per_layer,
            call=None if w.name.startswith("decode") else
            ("ss_fwd with the binding's cached workspace (C ABI ss_fwd_ws)" if args.workspace else "ss_fwd (C ABI)")),
        "hbm_gbs": alg_bytes(w) / (ms_step / 1e3) / 1e9,
        "gpu_launches": args.steps * res["launches"],
        "clocks": res["clocks"], "roofline": roof,
    }
    if res["e2e"] is not None:
        e = res["e2e"]
        out["e2e"] = {"value": units * world / (e["ms"] / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"], "ms_per_step": e["ms"],
                      "call": "ss_fwd_host (C ABI, pinned host buffers)"}
    if rank == 0 and not args.no_cpu_baseline:
        rate, passes, elapsed, cores = oracle_time(w)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": f"{passes} full pass(es) of the {w.name} workload, "
                                         f"{elapsed:.1f} s of fp64 oracle time"}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
