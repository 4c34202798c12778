"""Seeded synthetic inputs for the selective scan, shaped like Mamba layers.

This module draws random numbers and nothing else: it holds none of the
scan's arithmetic and imports nothing from the rest of the package, so the
CUDA path and the fp64 oracle can both be fed from it.

Recipe (per workload; draws are fp32, then cast to the I/O dtype):
  x, z            ~ N(0, 1)                        shape (batch, seqlen, dim)
  delta_raw       ~ N(0, 1)                        shape (batch, seqlen, dim)
  delta_bias[d]   = log(expm1(U[lo, hi]))          shape (dim,)   (inverse softplus
                                                   of a uniform step size)
  B, C            ~ N(0, 1)                        shape (batch, seqlen, dstate)
  D[d]            ~ N(0, 1)                        shape (dim,)
  A[d, n]         = -exp(A_log[d, n]),  A_log[d, n] = log(n + 1)  (or U[-1, 3]
                                                   for the random-A robustness case)
Draw order: x, z, delta_raw, bias uniform, B, C, D.  A, D and delta_bias are
always fp32; x, delta, z, B, C follow the I/O dtype.

Causal conv in front of the scan (own seeded stream, all fp32), the default
initialisation of a depthwise Conv1d layer with K taps (fan-in K):
  conv_w[d, k]    ~ U[-1/sqrt(K), 1/sqrt(K)]       shape (dim, K)
  conv_bias[d]    ~ U[-1/sqrt(K), 1/sqrt(K)]       shape (dim,)
  conv_state      ~ N(0, 1)                        shape (batch, dim, K-1)

Selection projections (own seeded stream; bf16), the default initialisation
of the two linear layers (fan-in dim and R):
  x               ~ N(0, 1)                        shape (batch, seqlen, dim)
  W_x[j, k]       ~ U[-1/sqrt(dim), 1/sqrt(dim)]   shape (R + 2N, dim)
  W_dt[d, r]      ~ U[-1/sqrt(R), 1/sqrt(R)]       shape (dim, R)

On ``device="cpu"`` the draws come from numpy's PCG64 stream (bit-identical on
every machine).  On a CUDA device they come from torch's device generator,
which is much faster for the multi-GB workloads; both are seeded.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    io: str                 # "f32" or "bf16"
    seed: int
    dt_lo: float = 1e-3     # uniform range of the step size behind delta_bias
    dt_hi: float = 1e-1
    random_A: bool = False
    with_z: bool = True
    with_D: bool = True
    with_bias: bool = True
    init_state: bool = False

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen * self.dim

    @property
    def items(self) -> int:
        return self.tokens * self.dstate

    def io_bytes(self) -> int:
        """Bytes of x, delta, z, B, C read plus out written (the compulsory traffic)."""
        e = 4 if self.io == "f32" else 2
        n_tok_tensors = 2 + (1 if self.with_z else 0) + 1   # x, delta, [z], out
        return e * (n_tok_tensors * self.tokens + 2 * self.batch * self.seqlen * self.dstate)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    io: str
    seed: int
    dt_lo: float = 1e-3
    dt_hi: float = 1e-1

    def step_bytes(self) -> int:
        """Per step: fp32 state read + written, x/delta/z read and out written (io),
        B and C read (io)."""
        e = 4 if self.io == "f32" else 2
        return (2 * 4 * self.batch * self.dim * self.dstate + 4 * e * self.batch * self.dim
                + 2 * e * self.batch * self.dstate)


# The five workloads: a tiny fp32 case, three Mamba-shaped prefill layers
# (130M: d_model 768 x expand 2; 1.4B: d_model 2048 x expand 2; a 256k-token
# long sequence) and a decode step.
TINY = ScanWorkload("tiny-f32-b1-l64-d16-n4", 1, 64, 16, 4, "f32", 0)
MAMBA_130M = ScanWorkload("mamba130m-bf16-b8-l2048-d1536-n16", 8, 2048, 1536, 16, "bf16", 1)
MAMBA_1P4B = ScanWorkload("mamba1.4b-bf16-b4-l8192-d4096-n16", 4, 8192, 4096, 16, "bf16", 2)
LONG_SEQ = ScanWorkload("long-bf16-b1-l262144-d2048-n16", 1, 262144, 2048, 16, "bf16", 3,
                        dt_lo=1e-4, dt_hi=1e-2)
DECODE = DecodeWorkload("decode-bf16-b256-d5120-n16-x128", 256, 5120, 16, 128, "bf16", 4)

SCAN_WORKLOADS = (TINY, MAMBA_130M, MAMBA_1P4B, LONG_SEQ)


def io_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


class _Draw:
    """One seeded stream: numpy PCG64 on the host, torch's generator on a GPU."""

    def __init__(self, seed: int, device: str):
        self.device = torch.device(device)
        if self.device.type == "cpu":
            self.rng = np.random.Generator(np.random.PCG64(seed))
        else:
            self.gen = torch.Generator(device=self.device)
            self.gen.manual_seed(seed)

    def normal(self, shape) -> torch.Tensor:
        if self.device.type == "cpu":
            return torch.from_numpy(self.rng.standard_normal(size=shape, dtype=np.float32))
        return torch.randn(shape, generator=self.gen, device=self.device, dtype=torch.float32)

    def uniform(self, shape, lo: float, hi: float) -> torch.Tensor:
        if self.device.type == "cpu":
            return torch.from_numpy(self.rng.uniform(lo, hi, size=shape))  # fp64
        u = torch.rand(shape, generator=self.gen, device=self.device, dtype=torch.float64)
        return lo + (hi - lo) * u


def make_scan_inputs(w: ScanWorkload, device: str = "cpu") -> dict:
    """Draw one scan problem.  Returns a dict of tensors on ``device``:
    x, delta, z (or None), A, B, C, D (or None), delta_bias (or None),
    initial_state (or None)."""
    g = _Draw(w.seed, device)
    dt = io_dtype(w.io)
    shape = (w.batch, w.seqlen, w.dim)
    x = g.normal(shape).to(dt)
    z = g.normal(shape).to(dt) if w.with_z else None
    delta = g.normal(shape).to(dt)
    u = g.uniform((w.dim,), w.dt_lo, w.dt_hi)
    bias = torch.log(torch.expm1(u)).to(torch.float32) if w.with_bias else None
    Bm = g.normal((w.batch, w.seqlen, w.dstate)).to(dt)
    Cm = g.normal((w.batch, w.seqlen, w.dstate)).to(dt)
    D = g.normal((w.dim,)) if w.with_D else None
    if w.random_A:
        a_log = g.uniform((w.dim, w.dstate), -1.0, 3.0)
    else:
        a_log = torch.log(torch.arange(1, w.dstate + 1, dtype=torch.float64,
                                       device=g.device)).expand(w.dim, w.dstate)
    A = (-torch.exp(a_log)).to(torch.float32).contiguous()
    h0 = g.normal((w.batch, w.dim, w.dstate)) if w.init_state else None
    return dict(x=x, delta=delta, z=z, A=A, B=Bm, C=Cm, D=D, delta_bias=bias, initial_state=h0)


def make_decode_inputs(w: DecodeWorkload, device: str = "cpu") -> dict:
    """Draw a chained decode problem: the initial fp32 state ~ N(0,1) and, for
    each of ``w.steps`` steps, x, delta, z (batch, dim) and B, C (batch, dstate)."""
    g = _Draw(w.seed, device)
    dt = io_dtype(w.io)
    tok = (w.steps, w.batch, w.dim)
    x = g.normal(tok).to(dt)
    z = g.normal(tok).to(dt)
    delta = g.normal(tok).to(dt)
    u = g.uniform((w.dim,), w.dt_lo, w.dt_hi)
    bias = torch.log(torch.expm1(u)).to(torch.float32)
    Bm = g.normal((w.steps, w.batch, w.dstate)).to(dt)
    Cm = g.normal((w.steps, w.batch, w.dstate)).to(dt)
    D = g.normal((w.dim,))
    a_log = torch.log(torch.arange(1, w.dstate + 1, dtype=torch.float64,
                                   device=g.device)).expand(w.dim, w.dstate)
    A = (-torch.exp(a_log)).to(torch.float32).contiguous()
    state = g.normal((w.batch, w.dim, w.dstate))
    return dict(state=state, x=x, delta=delta, z=z, A=A, B=Bm, C=Cm, D=D, delta_bias=bias)


def make_conv_inputs(batch: int, dim: int, width: int, seed: int, device: str = "cpu",
                     with_bias: bool = True, with_state: bool = False) -> dict:
    """Draw the causal conv's parameters (and optionally its history):
    conv_w (dim, width), conv_bias (dim,) or None, conv_state (batch, dim,
    width-1) or None; all fp32."""
    g = _Draw(seed, device)
    bound = 1.0 / float(width) ** 0.5
    w = g.uniform((dim, width), -bound, bound).to(torch.float32).contiguous()
    bias = g.uniform((dim,), -bound, bound).to(torch.float32) if with_bias else None
    state = g.normal((batch, dim, width - 1)).contiguous() if with_state else None
    return dict(conv_w=w, conv_bias=bias, conv_state=state)


def make_proj_inputs(batch: int, seqlen: int, dim: int, dt_rank: int, dstate: int, seed: int,
                     device: str = "cpu") -> dict:
    """Draw x and the two projection weights, bf16."""
    g = _Draw(seed, device)
    x = g.normal((batch, seqlen, dim)).to(torch.bfloat16)
    bx = 1.0 / float(dim) ** 0.5
    bd = 1.0 / float(dt_rank) ** 0.5
    W_x = g.uniform((dt_rank + 2 * dstate, dim), -bx, bx).to(torch.bfloat16).contiguous()
    W_dt = g.uniform((dim, dt_rank), -bd, bd).to(torch.bfloat16).contiguous()
    return dict(x=x, W_x=W_x, W_dt=W_dt)
