"""Sequence parallelism for the forward scan: one sequence cut into contiguous segments, one
segment per rank of a process group, with a single exchange between two passes.

The carry that "mamba-metal: Apple Silicon で Mamba を動かす" (section "チャンク間 running
prefix") hands from one chunk to the next is handed here from one rank's segment to the next:

  1. every rank summarises its segment: the state its steps leave from a zero start, h_end, and
     the sum of its Δ (ss_fwd_summary; the decay across the segment is exp(A · Σ Δ));
  2. the ranks all-gather the summaries (the only exchange: batch·Dm·(N + 1) floats per rank)
     and each composes them left to right into the state entering its own segment
     (ss_carry_compose: H_0 = h0, H_s = exp(A · Σ Δ_{s-1}) · H_{s-1} + h_end_{s-1});
  3. every rank runs its segment from that state (ss_fwd_h0), giving its part of y and, on the
     last rank, the sequence's final state.

Every step of the arithmetic runs in the library's kernels; this module only moves tensors and
calls the collective.  With the gloo backend the summaries travel through host memory (gloo
does not take CUDA tensors); with NCCL they stay on the device.
"""
from __future__ import annotations


class LibraryOps:
    """The three device calls of the scheme, through the C ABI (the default)."""

    def summary(self, u, delta_raw, delta_bias, A_log, B):
        from . import ss_fwd_summary
        return ss_fwd_summary(u, delta_raw, delta_bias, A_log, B)

    def compose(self, slots, dsum, A_log, h0):
        from . import ss_carry_compose
        return ss_carry_compose(slots, dsum, A_log, h0=h0)

    def fwd_h0(self, u, delta_raw, delta_bias, A_log, B, C, D, z, h0, last_state, workspace):
        from . import ss_fwd
        return ss_fwd(u, delta_raw, delta_bias, A_log, B, C, D, z, last_state=last_state, h0=h0,
                      workspace=workspace)


def _all_gather(t, group):
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if dist.get_backend(group) == "gloo" and t.is_cuda:
        host = t.detach().cpu()
        parts = [torch.empty_like(host) for _ in range(world)]
        dist.all_gather(parts, host, group=group)
        return [p.to(t.device) for p in parts]
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return parts


def ss_fwd_seqpar(u, delta_raw, delta_bias, A_log, B, C, D=None, z=None, h0=None, last_state=None,
                  group=None, workspace=True, ops=None):
    """This rank's part of a forward scan whose sequence is split across the ranks of `group`
    in rank order (rank r holds steps [t_r, t_{r+1}) of u, delta_raw, z, B, C; segment lengths
    may differ).  h0 is the state before the first segment and must be the same tensor value on
    every rank (None: zeros).  Returns y for this rank's steps; last_state (if given) receives
    the state after this rank's segment, on the last rank the sequence's final state.
    `ops` replaces the three device calls (for tests of the exchange without a GPU)."""
    import torch
    import torch.distributed as dist
    ops = ops or LibraryOps()
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    h_end, dsum = ops.summary(u, delta_raw, delta_bias, A_log, B)
    ends = _all_gather(h_end, group)
    sums = _all_gather(dsum, group)
    batch, Dm, N = h_end.shape
    # slot s (s >= 1) holds the end state of segment s - 1; slot 0 receives h0 (or zeros)
    slots = torch.empty((world, batch, Dm, N), dtype=h_end.dtype, device=h_end.device)
    for s in range(1, world):
        slots[s].copy_(ends[s - 1])
    dstack = torch.stack(sums[: world - 1]) if world > 1 else None
    ops.compose(slots, dstack, A_log, h0)
    h_in = slots[rank].contiguous()
    return ops.fwd_h0(u, delta_raw, delta_bias, A_log, B, C, D, z, h_in, last_state, workspace)
