"""The cross-rank exchange of sequence parallelism (selective_state_space_scan_gb300.seqpar),
tested without a GPU: gloo ranks on the CPU, each holding one segment of one sequence, with
the three device calls replaced by oracle-backed stand-ins, so that what is checked is the
exchange itself (which summaries are gathered, in which order, which slot each rank takes).
The concatenated outputs must equal one fp64 oracle call over the whole sequence.

The stand-ins: the summary is the oracle's end state from a zero start plus Σ softplus(δ + bias);
the composition applies H_s = exp(A · Σ Δ_{s-1}) · H_{s-1} + h_end_{s-1} written out in numpy
(the carry of "mamba-metal: Apple Silicon で Mamba を動かす", section "チャンク間 running
prefix"); the segment pass is the oracle from the given initial state.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from selective_state_space_scan_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """CPU stand-ins for the three device calls, on float64 torch tensors."""

    def summary(self, u, delta_raw, delta_bias, A_log, B):
        import torch
        import oracle
        f = lambda t: None if t is None else t.numpy()
        batch, L, Dm = u.shape
        N = A_log.shape[1]
        zeros = np.zeros((batch, L, N), np.float32)
        _, last, _ = oracle.ss_fwd(f(u), f(delta_raw), f(delta_bias), f(A_log), f(B), zeros, None, None)
        bias = np.zeros(Dm) if delta_bias is None else f(delta_bias).astype(np.float64)
        sp = np.vectorize(oracle.softplus)(f(delta_raw).astype(np.float64) + bias)
        return torch.from_numpy(np.ascontiguousarray(last)), torch.from_numpy(sp.sum(axis=1))

    def compose(self, slots, dsum, A_log, h0):
        A = -np.exp(A_log.numpy().astype(np.float64))             # [Dm, N]
        s = slots.numpy()
        s[0] = 0.0 if h0 is None else h0.numpy()
        for k in range(1, s.shape[0]):
            decay = np.exp(A[None, :, :] * dsum.numpy()[k - 1][:, :, None])
            s[k] = decay * s[k - 1] + s[k]
        return slots

    def fwd_h0(self, u, delta_raw, delta_bias, A_log, B, C, D, z, h0, last_state, workspace):
        import torch
        import oracle
        f = lambda t: None if t is None else t.numpy()
        y, last, _ = oracle.ss_fwd(f(u), f(delta_raw), f(delta_bias), f(A_log), f(B), f(C), f(D), f(z),
                                   h0=h0.numpy())
        if last_state is not None:
            last_state.copy_(torch.from_numpy(last))
        return torch.from_numpy(y)


def _rank_main(rank, world, port, cuts, out):
    import torch
    import torch.distributed as dist
    from selective_state_space_scan_gb300.seqpar import ss_fwd_seqpar
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.fwd_inputs(2, cuts[-1], 24, 16, seed=77)
    a = w.arrays
    t0, t1 = cuts[rank], cuts[rank + 1]
    seg = lambda x: torch.from_numpy(np.ascontiguousarray(x[:, t0:t1]))
    whole = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x))
    h0 = torch.from_numpy(synth.initial_state(2, 24, 16, seed=78).astype(np.float64))
    last = torch.empty((2, 24, 16), dtype=torch.float64)
    y = ss_fwd_seqpar(seg(a["u"]), seg(a["delta_raw"]), whole(a["delta_bias"]), whole(a["A_log"]), seg(a["B"]),
                      seg(a["C"]), whole(a["D"]), seg(a["z"]), h0=h0, last_state=last, ops=OracleOps())
    out.put((rank, y.numpy(), last.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [(0, 150, 300), (0, 1, 170, 300)], ids=["2-ranks", "3-ranks-uneven"])
def test_seqpar_exchange_matches_one_call(cuts):
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    import oracle
    world = len(cuts) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, cuts, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.fwd_inputs(2, cuts[-1], 24, 16, seed=77)
    a = w.arrays
    h0 = synth.initial_state(2, 24, 16, seed=78).astype(np.float64)
    ref_y, ref_last, _ = oracle.ss_fwd(a["u"], a["delta_raw"], a["delta_bias"], a["A_log"], a["B"], a["C"],
                                       a["D"], a["z"], h0=h0)
    y = np.concatenate([r[1] for r in res], axis=1)
    np.testing.assert_allclose(y, ref_y, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(res[-1][2], ref_last, rtol=1e-9, atol=1e-10)
    # every rank's last_state is the sequence's state after that rank's segment
    for rank, _, last in res[:-1]:
        t1 = cuts[rank + 1]
        _, ref_mid, _ = oracle.ss_fwd(a["u"][:, :t1], a["delta_raw"][:, :t1], a["delta_bias"], a["A_log"],
                                      a["B"][:, :t1], a["C"][:, :t1], a["D"], a["z"][:, :t1], h0=h0)
        np.testing.assert_allclose(last, ref_mid, rtol=1e-9, atol=1e-10)
