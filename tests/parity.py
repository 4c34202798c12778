"""Helpers for the GPU-vs-oracle parity tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Elementwise bound |y - y_ref| <= tol * (1 + |y_ref|), for outputs and states.
TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}


def f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def to_device(inp: dict, dev) -> dict:
    return {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}


def oracle_full(inp: dict, delta_softplus=True):
    return oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                           f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                           delta_bias=f64(inp["delta_bias"]), delta_softplus=delta_softplus,
                           initial_state=f64(inp["initial_state"]))


def sample_channels(bsz, dim, per_batch=6, seed=0, max_batches=4):
    """(b, [d...]) pairs: the edge channels and a few random ones."""
    r = np.random.default_rng(seed)
    bs = sorted(set([0, bsz - 1] + list(r.integers(0, bsz, size=max(0, max_batches - 2)))))
    out = []
    for b in bs:
        ds = {0, dim - 1, dim // 2}
        ds |= set(int(v) for v in r.integers(0, dim, size=max(0, per_batch - len(ds))))
        out.append((int(b), sorted(ds)))
    return out


def oracle_sampled(inp: dict, samples, delta_softplus=True):
    """Oracle outputs for sampled channels only.  Returns {b: (ds, out (L, nd), last (nd, N))}."""
    res = {}
    for b, ds in samples:
        idx = torch.tensor(ds, device=inp["x"].device)
        g = lambda t: None if t is None else f64(t[b].index_select(-1, idx))[None]  # (1, L, nd)
        vec = lambda t: None if t is None else f64(t.index_select(0, idx))
        h0 = None if inp["initial_state"] is None else f64(inp["initial_state"][b].index_select(0, idx))[None]
        out, last = oracle.scan_fwd(g(inp["x"]), g(inp["delta"]), f64(inp["A"].index_select(0, idx)),
                                    f64(inp["B"][b])[None], f64(inp["C"][b])[None], D=vec(inp["D"]),
                                    z=g(inp["z"]), delta_bias=vec(inp["delta_bias"]),
                                    delta_softplus=delta_softplus, initial_state=h0)
        res[b] = (ds, out[0], last[0])
    return res
