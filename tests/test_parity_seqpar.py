"""Sequence parallelism on the GPU: the segment summary (ss_fwd_summary), the left-to-right
composition of summaries (ss_carry_compose) and the whole cross-rank scheme with two gloo ranks.

The two ranks are two processes that both use this one GPU; no kernel of one waits on the
other: the summaries travel through host memory between the two processes' launches (the
gloo all-gather), so each process's kernels only ever wait on their own stream.
"""
import os
import socket

import numpy as np
import pytest

import oracle
import selective_state_space_scan_gb300 as ss
from selective_state_space_scan_gb300 import synth

from helpers import FP32_REL_L2, BF16_REL_L2, assert_fwd_close, f32dev, rel_l2, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert ss.device_error(clear=True) == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 63, 64, 65, 1000])
def test_summary_against_oracle(io, L):
    """h_end is the oracle's final state from a zero start; dsum the sum of softplus(δ + bias)."""
    w = synth.fwd_inputs(3, L, 72, 16, io=io, seed=500 + L)      # rows of whole 16-byte units (TMA)
    a = w.arrays
    h_end, dsum = ss.ss_fwd_summary(to_dev(a["u"], io), to_dev(a["delta_raw"], io), f32dev(a["delta_bias"]),
                                    f32dev(a["A_log"]), to_dev(a["B"], io))
    torch.cuda.synchronize()
    _, ref_last, _ = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"], a["D"],
                                   a["z"])
    ref_dsum = np.vectorize(oracle.softplus)(a["delta_raw"].astype(np.float64) +
                                             a["delta_bias"].astype(np.float64)).sum(axis=1)
    tol = FP32_REL_L2 if io == "f32" else 1e-4
    assert rel_l2(to_host(h_end), ref_last) <= tol
    assert rel_l2(to_host(dsum), ref_dsum) <= 1e-5


def test_summary_empty_and_refusals():
    w = synth.fwd_inputs(2, 10, 40, 16, seed=510)
    a = w.arrays
    h_end = torch.full((2, 40, 16), 7.0, device="cuda")
    dsum = torch.full((2, 40), 7.0, device="cuda")
    ss.ss_fwd_summary(to_dev(a["u"][:, :0], "f32"), to_dev(a["delta_raw"][:, :0], "f32"), f32dev(a["delta_bias"]),
                      f32dev(a["A_log"]), to_dev(a["B"][:, :0], "f32"), h_end=h_end, dsum=dsum)
    torch.cuda.synchronize()
    assert torch.all(h_end == 0) and torch.all(dsum == 0)
    # B rows of 5 states cannot be TMA-fed: refused, no fallback
    w5 = synth.fwd_inputs(1, 10, 40, 5, seed=511)
    b = w5.arrays
    with pytest.raises(ss.SelscanError):
        ss.ss_fwd_summary(to_dev(b["u"], "f32"), to_dev(b["delta_raw"], "f32"), f32dev(b["delta_bias"]),
                          f32dev(b["A_log"]), to_dev(b["B"], "f32"))


@pytest.mark.parametrize("nseg", [1, 2, 5])
def test_compose_then_segments_equal_one_call(nseg):
    """Summaries of nseg segments, composed, then each segment run from its entering state: the
    concatenation equals one call over the whole sequence (against the oracle), for fp32 and
    from a nonzero h0."""
    L, batch, Dm, N = 600, 2, 96, 16
    w = synth.fwd_inputs(batch, L, Dm, N, seed=520 + nseg)
    a = w.arrays
    h0 = synth.initial_state(batch, Dm, N, seed=521)
    cuts = np.linspace(0, L, nseg + 1).astype(int)
    seg = lambda x, s: to_dev(np.ascontiguousarray(x[:, cuts[s]:cuts[s + 1]]), "f32")
    slots = torch.empty((nseg, batch, Dm, N), device="cuda")
    dsums = torch.empty((max(nseg - 1, 1), batch, Dm), device="cuda")
    for s in range(nseg - 1):
        h_end, dsum = ss.ss_fwd_summary(seg(a["u"], s), seg(a["delta_raw"], s), f32dev(a["delta_bias"]),
                                        f32dev(a["A_log"]), seg(a["B"], s))
        slots[s + 1].copy_(h_end)
        dsums[s].copy_(dsum)
    ss.ss_carry_compose(slots, dsums[: nseg - 1] if nseg > 1 else None, f32dev(a["A_log"]), h0=f32dev(h0))
    ys, last = [], None
    for s in range(nseg):
        last = torch.empty((batch, Dm, N), device="cuda")
        ys.append(ss.ss_fwd(seg(a["u"], s), seg(a["delta_raw"], s), f32dev(a["delta_bias"]), f32dev(a["A_log"]),
                            seg(a["B"], s), seg(a["C"], s), f32dev(a["D"]), seg(a["z"], s), last_state=last,
                            h0=slots[s].contiguous()))
    torch.cuda.synchronize()
    y = np.concatenate([to_host(t) for t in ys], axis=1)
    ref_y, ref_last, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"],
                                         a["D"], a["z"], h0=h0.astype(np.float64))
    assert_fwd_close("f32", y, ref_y, mag, to_host(last), ref_last, what=f"compose nseg={nseg}")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, io, cuts, out):
    import torch
    import torch.distributed as dist
    import selective_state_space_scan_gb300 as ss
    from selective_state_space_scan_gb300.seqpar import ss_fwd_seqpar
    from helpers import f32dev, to_dev, to_host
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    w = synth.fwd_inputs(2, cuts[-1], 160, 16, io=io, seed=530)
    a = w.arrays
    t0, t1 = cuts[rank], cuts[rank + 1]
    seg = lambda x: to_dev(np.ascontiguousarray(x[:, t0:t1]), io)
    last = torch.empty((2, 160, 16), device="cuda")
    y = ss_fwd_seqpar(seg(a["u"]), seg(a["delta_raw"]), f32dev(a["delta_bias"]), f32dev(a["A_log"]), seg(a["B"]),
                      seg(a["C"]), f32dev(a["D"]), seg(a["z"]), last_state=last)
    torch.cuda.synchronize()
    err = ss.device_error(clear=True)
    out.put((rank, to_host(y), to_host(last), err))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_two_ranks_gloo_match_one_call(io):
    """Two processes, each holding half of the sequence, exchange their summaries over gloo and
    run their halves; the concatenated y and the last rank's final state equal the oracle's
    single call over the whole sequence."""
    import torch.multiprocessing as mp
    cuts = (0, 700, 1500)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, io, cuts, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(2)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert all(r[3] == 0 for r in res)
    w = synth.fwd_inputs(2, cuts[-1], 160, 16, io=io, seed=530)
    a = w.arrays
    ref_y, ref_last, mag = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"],
                                         a["D"], a["z"])
    y = np.concatenate([r[1] for r in res], axis=1)
    assert_fwd_close(io, y, ref_y, mag, res[1][2], ref_last, what=f"seqpar 2 ranks {io}")
