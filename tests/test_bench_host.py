"""Host-side pieces of bench.py that need no GPU: the multi-rank timing aggregation over a
2-rank gloo group, the whole-job throughput, the algorithmic byte counts, the lookup of
stored DRAM traffic, the clocks summary and the oracle reference arm."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from selective_state_space_scan_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(10.0 + rank, dist)          # rank 1 is the slower one
    value = bench.job_throughput(1000, world, slowest, steps=4)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in res:
        assert slowest == 11.0                                  # max over ranks, on every rank
        assert value == pytest.approx(1000 * 2 / (11.0e-3 / 4))


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_algorithmic_bytes_match_the_formula():
    w = synth.Workload("mamba130m", 8, 2048, 1536, 16, "f32", 1)
    assert bench.alg_bytes(w) == 405_647_360
    w = synth.Workload("long32k", 1, 32768, 1536, 16, "f32", 2)
    assert bench.alg_bytes(w) == 809_709_568
    w = synth.Workload("mamba2p8b_bf16", 4, 8192, 5120, 16, "bf16", 3)
    assert bench.alg_bytes(w) == 1_345_953_792
    w = synth.Workload("decode1p4b", 64, 1, 4096, 16, "f32", 4)
    assert bench.alg_bytes(w) == 48 * 38_035_456


def test_measured_traffic_follows_the_sources(tmp_path, monkeypatch):
    """Stored DRAM traffic is reported only for the kernel it was captured on and only while
    the hash of that kernel's sources matches; a second call of a workload has its own
    "workload:kernel" record."""
    import json
    csrc = tmp_path / "selective_state_space_scan_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in set(sum(bench.KERNEL_SOURCES.values(), ())):
        (csrc / f).write_text("// " + f + "\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    lane, seg = "ss_fwd_lane_kernel(lpc=4)", "ss_fwd_seg_kernel"
    tab = {"wl": {"kernel": lane, "source_hash": bench.kernel_source_hash(lane), "dram_bytes_per_launch": 1.0},
           "wl:" + seg: {"kernel": seg, "source_hash": bench.kernel_source_hash(seg), "dram_bytes_per_launch": 2.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(tab))
    assert bench.measured_traffic("wl", lane) == 1.0
    assert bench.measured_traffic("wl", seg) == 2.0
    assert bench.measured_traffic("wl", "ss_step_kernel") is None
    assert bench.measured_traffic("other", lane) is None
    # a segment-kernel source changes: its record goes stale, the lane kernel's does not
    (csrc / "ss_fwd_seg.cuh").write_text("// changed\n")
    assert bench.measured_traffic("wl", seg) is None
    assert bench.measured_traffic("wl", lane) == 1.0
    # a source both kernels are built from changes: both go stale
    (csrc / "fwd_configs.h").write_text("// changed\n")
    assert bench.measured_traffic("wl", lane) is None


def _bench(args, env_extra):
    import json
    import subprocess
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_runs_the_oracle_on_the_host():
    """bench.py --impl reference: the oracle timed on the host cores, one JSON line on rank 0
    carrying the contract's keys, nothing from any other rank."""
    args = ["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"]
    out = _bench(args, {"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert len(out) == 1
    d = out[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")
    assert _bench(args, {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_clock_summary_reads_nvidia_smi_rows(tmp_path):
    """The clocks object from nvidia-smi's CSV rows: median SM clock over the loaded samples,
    the maximum clock, and each throttle reason seen Active in any sample."""
    rows = ["0, 1965, 2070, 410.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 2055, 2070, 890.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 345, 2070, 120.0, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active",   # idle
            "garbage line"]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    c = bench.ClockSampler(0)
    c.path = str(path)
    c.warmup_steps = 12
    s = c.summary()
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0        # idle sample left out of the median
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 4 and s["warmup_steps_run"] == 12
    path.write_text(rows[0].replace("Not Active, Not Active, Not Active, Not Active",
                                    "Active, Not Active, Active, Not Active") + "\n")
    c.path = str(path)
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.path = str(tmp_path / "empty.csv")
    (tmp_path / "empty.csv").write_text("")
    assert c.summary()["reasons"] == ["unavailable"]
