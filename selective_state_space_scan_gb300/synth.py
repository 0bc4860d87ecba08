"""Seeded synthetic inputs shaped like the pages' selective-scan workloads.

This module draws random numbers and converts them to the storage types the
library takes; it holds none of the scan's arithmetic.  Both the CUDA path (via the
tests and the benchmark) and the fp64 oracle consume the arrays it returns, so the
two sides always see identical values.

Generator: numpy's Philox-4x32-10 counter-based bit generator (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011), seeded through a
SeedSequence; normals come from numpy's ziggurat sampler.

Draw order for a forward workload: u, delta_raw, z, B, C, delta_bias, D.
For a decode workload: x, delta_raw, z, B, C, delta_bias, D, state.

bf16 inputs are drawn in fp32 and rounded to the nearest bf16 (ties to even); the
fp32 arrays then hold exactly the bf16 values, and the uint16 bit patterns are kept
for upload.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), int(stream)])))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array holding the bf16-rounded values of x."""
    return bf16_to_f32(bf16_bits(x))


@dataclass
class Workload:
    """One forward (or decode) problem.  `arrays` holds float32 numpy arrays with the
    exact values both sides consume; `io` is "f32" or "bf16" (the storage type of
    u/x, delta_raw, z, B, C and y; parameters and state are always fp32)."""
    name: str
    batch: int
    L: int
    Dm: int
    N: int
    io: str
    seed: int
    arrays: Dict[str, Optional[np.ndarray]] = field(default_factory=dict)

    @property
    def state_updates(self) -> int:
        return self.batch * self.L * self.Dm * self.N

    def io_bytes(self) -> int:
        return 2 if self.io == "bf16" else 4


# The five workloads: (batch, L, Dm, N, io, distribution, seed).
CONFIGS = {
    "tiny": dict(batch=1, L=64, Dm=16, N=4, io="f32", dist="tiny", seed=0),
    "mamba130m": dict(batch=8, L=2048, Dm=1536, N=16, io="f32", dist="mamba", seed=1),
    "long32k": dict(batch=1, L=32768, Dm=1536, N=16, io="f32", dist="mamba", seed=2),
    "mamba2p8b_bf16": dict(batch=4, L=8192, Dm=5120, N=16, io="bf16", dist="mamba", seed=3),
    "decode1p4b": dict(batch=64, L=1, Dm=4096, N=16, io="f32", dist="decode", seed=4),
}


def _io_cast(x: np.ndarray, io: str) -> np.ndarray:
    x = x.astype(np.float32, copy=False)
    return round_bf16(x) if io == "bf16" else x


def fwd_inputs(batch: int, L: int, Dm: int, N: int, io: str = "f32", seed: int = 0,
               dist: str = "mamba", with_z: bool = True, with_D: bool = True,
               with_bias: bool = True, name: str = "custom") -> Workload:
    """Forward-scan inputs.

    dist="mamba": u, z ~ N(0,1); delta_raw ~ N(-4,1); delta_bias[d] ~ U(-1,0);
                  A_log[d,n] = log(n+1); B, C ~ N(0,1); D ~ N(1, 0.1)  (0.1 is the sd).
    dist="tiny":  u, z, delta_raw ~ N(0,1); delta_bias = 0.1; A_log = log(n+1);
                  B, C ~ N(0,1); D = 1.
    """
    g = rng_for(seed)
    f = np.float32
    if dist == "mamba":
        u = g.standard_normal((batch, L, Dm), dtype=f)
        delta_raw = g.standard_normal((batch, L, Dm), dtype=f) - f(4.0)
        z = g.standard_normal((batch, L, Dm), dtype=f)
        B = g.standard_normal((batch, L, N), dtype=f)
        C = g.standard_normal((batch, L, N), dtype=f)
        bias = g.uniform(-1.0, 0.0, size=Dm).astype(f)
        D = (f(1.0) + f(0.1) * g.standard_normal(Dm, dtype=f)).astype(f)
    elif dist == "tiny":
        u = g.standard_normal((batch, L, Dm), dtype=f)
        delta_raw = g.standard_normal((batch, L, Dm), dtype=f)
        z = g.standard_normal((batch, L, Dm), dtype=f)
        B = g.standard_normal((batch, L, N), dtype=f)
        C = g.standard_normal((batch, L, N), dtype=f)
        bias = np.full(Dm, 0.1, f)
        D = np.ones(Dm, f)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    A_log = np.tile(np.log(np.arange(1, N + 1, dtype=np.float64)).astype(f), (Dm, 1))
    arrays = dict(u=_io_cast(u, io), delta_raw=_io_cast(delta_raw, io),
                  z=_io_cast(z, io) if with_z else None,
                  B=_io_cast(B, io), C=_io_cast(C, io),
                  delta_bias=bias if with_bias else None, D=D if with_D else None,
                  A_log=np.ascontiguousarray(A_log))
    return Workload(name, batch, L, Dm, N, io, seed, arrays)


def step_inputs(batch: int, Dm: int, N: int, io: str = "f32", seed: int = 4, layer: int = 0,
                with_z: bool = True, with_bias: bool = False, name: str = "decode") -> Workload:
    """Decode-step inputs for one layer: state h ~ N(0, 0.5) (sd 0.5); x, z, delta_raw ~ N(0,1);
    B, C [batch, N] ~ N(0,1); A_log = log(n+1); D = 1; delta_bias = 0 (absent) unless asked."""
    g = rng_for(seed, layer)
    f = np.float32
    x = g.standard_normal((batch, Dm), dtype=f)
    delta_raw = g.standard_normal((batch, Dm), dtype=f)
    z = g.standard_normal((batch, Dm), dtype=f)
    B = g.standard_normal((batch, N), dtype=f)
    C = g.standard_normal((batch, N), dtype=f)
    bias = g.uniform(-1.0, 0.0, size=Dm).astype(f)
    D = np.ones(Dm, f)
    state = (f(0.5) * g.standard_normal((batch, Dm, N), dtype=f)).astype(f)
    A_log = np.tile(np.log(np.arange(1, N + 1, dtype=np.float64)).astype(f), (Dm, 1))
    arrays = dict(x=_io_cast(x, io), delta_raw=_io_cast(delta_raw, io),
                  z=_io_cast(z, io) if with_z else None, B=_io_cast(B, io), C=_io_cast(C, io),
                  delta_bias=bias if with_bias else None, D=D, A_log=np.ascontiguousarray(A_log),
                  state=state)
    return Workload(name, batch, 1, Dm, N, io, seed, arrays)


def initial_state(batch: int, Dm: int, N: int, seed: int = 0) -> np.ndarray:
    """A forward pass's initial state h0 [batch, Dm, N] fp32 ~ N(0, 0.5) (sd 0.5), the
    distribution of the decode workload's states (its own generator stream)."""
    g = rng_for(seed, 3)
    f = np.float32
    return (f(0.5) * g.standard_normal((batch, Dm, N), dtype=f)).astype(f)


def config(name: str, **overrides) -> Workload:
    """The named workload (see CONFIGS); decode returns layer 0."""
    c = dict(CONFIGS[name])
    c.update(overrides)
    if c["dist"] == "decode":
        return step_inputs(c["batch"], c["Dm"], c["N"], c["io"], c["seed"], name=name)
    return fwd_inputs(c["batch"], c["L"], c["Dm"], c["N"], c["io"], c["seed"], c["dist"], name=name)
