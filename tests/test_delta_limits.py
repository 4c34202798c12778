"""GPU parity at the step size's limits, through every kernel family.

The step size Delta is the selection mechanism's gate ("Mamba的三大创新",
S4 -> S6 section, the step-size paragraph): a very small Delta keeps the
state and ignores the current token, a very large Delta resets the state to
the current token's input.  The oracle is pinned at both limits; these tests
drive the CUDA kernels there:

* Delta_raw = -1e4 with no bias: softplus gives Delta = 0 exactly, so the
  decay is exactly 1 and the input term exactly 0.  The final state must come
  back bit-identical to the initial state, and y = (C h0 + D x) silu(z).
* Delta_raw = +60 and +100: the large-input branch of softplus, and decays
  2^(Delta A log2 e) far below the smallest normal float (flushed to 0):
  h_t = Delta_t B_t x_t.
* exact zero-order hold with |Delta A| on both sides of 1/16, where the
  kernels switch between the series and the closed form of (e^{Delta A} - 1)/A.

Kernels: the one-warp tiled scan (dstate 16), the warp-specialised scan (the
exact-ZOH path), the general kernel (dstate 4, and an unaligned channel
count), and the decode step; fp32 and bf16 I/O; elementwise against the fp64
oracle with the forward's bounds.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu

BASE = synth.ScanWorkload("delta-limit", 2, 200, 48, 16, "bf16", 41, init_state=True)

# (name, workload changes): which kernel family each shape reaches
SHAPES = {
    "warp": dict(),                       # 16-byte rows, dstate 16: the one-warp tiled scan
    "generic_n4": dict(dstate=4),         # dstate 4: the general kernel
    "generic_unaligned": dict(dim=42),    # 84-byte bf16 rows: the general kernel
}


def set_delta(inp, value, frac=1.0, seed=0):
    """Delta_raw = value at a random fraction of the tokens (all if frac = 1),
    and no bias, so Delta = softplus(value) there."""
    d = inp["delta"]
    if frac >= 1.0:
        inp["delta"] = torch.full_like(d, value)
    else:
        r = np.random.default_rng(seed)
        mask = torch.from_numpy(r.random(tuple(d.shape)) < frac)
        inp["delta"] = torch.where(mask, torch.full_like(d, value), d)
    inp["delta_bias"] = torch.zeros_like(inp["delta_bias"])


def scan_both(inp, cuda, zoh=False):
    dev = to_device(inp, cuda)
    out, last = ops.scan_fwd(**dev, discretization="zoh" if zoh else "euler")
    torch.cuda.synchronize()
    ref, ref_last = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                                    f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                                    delta_bias=f64(inp["delta_bias"]),
                                    initial_state=f64(inp["initial_state"]), zoh=zoh)
    return out, last, ref, ref_last, dev


def plan_path(w):
    return binding.ssm_scan_plan(binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate,
                                                   synth.io_dtype(w.io))).path


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("zoh", [False, True])
def test_tiny_delta_keeps_the_state(cuda, io, shape, zoh):
    w = dataclasses.replace(BASE, io=io, name=f"tiny-{shape}-{io}", **SHAPES[shape])
    assert (plan_path(w) == 3) == (shape == "warp")
    inp = synth.make_scan_inputs(w)
    set_delta(inp, -1.0e4)
    out, last, ref, ref_last, dev = scan_both(inp, cuda, zoh)
    # decay exactly 1 and input term exactly 0: the state is returned unchanged
    assert torch.equal(last, dev["initial_state"])
    # the readout of the unchanged state: (C_t h0 + D x_t) silu(z_t)
    C = f64(inp["C"])
    h0 = f64(inp["initial_state"])
    zz = f64(inp["z"])
    expect = (np.einsum("btn,bdn->btd", C, h0) + f64(inp["D"]) * f64(inp["x"])) * zz / (1 + np.exp(-zz))
    assert rel_err(ref, expect) <= 1e-12               # the oracle at this limit
    assert rel_err(f64(out), ref) <= TOL[synth.io_dtype(io)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("value", [60.0, 100.0])
def test_large_delta_resets_the_state(cuda, io, shape, value):
    w = dataclasses.replace(BASE, io=io, name=f"large-{shape}-{io}", **SHAPES[shape])
    inp = synth.make_scan_inputs(w)
    set_delta(inp, value)
    out, last, ref, ref_last, _ = scan_both(inp, cuda)
    # the state after the last token is that token's input term alone
    x, B = f64(inp["x"])[:, -1], f64(inp["B"])[:, -1]
    dl = np.log1p(np.exp(-value)) + value
    assert rel_err(ref_last, dl * x[:, :, None] * B[:, None, :]) <= 1e-9
    tol = TOL[synth.io_dtype(io)]
    assert rel_err(f64(out), ref) <= tol
    assert rel_err(f64(last), ref_last) <= tol


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", ["warp", "generic_n4"])
def test_mixed_limits_in_one_sequence(cuda, io, shape):
    """Tokens at both limits scattered among ordinary ones: the state is held
    across Delta = 0 tokens and reset at Delta = 100 tokens, mid-sequence."""
    w = dataclasses.replace(BASE, io=io, seqlen=300, name=f"mixed-{shape}-{io}", **SHAPES[shape])
    inp = synth.make_scan_inputs(w)
    set_delta(inp, -1.0e4, frac=0.3, seed=1)
    d = inp["delta"]
    mask = torch.from_numpy(np.random.default_rng(2).random(tuple(d.shape)) < 0.05)
    inp["delta"] = torch.where(mask, torch.full_like(d, 100.0), d)
    inp["delta_bias"] = None
    out, last, ref, ref_last, _ = scan_both(inp, cuda)
    tol = TOL[synth.io_dtype(io)]
    assert rel_err(f64(out), ref) <= tol
    assert rel_err(f64(last), ref_last) <= tol


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", ["warp", "generic_n4"])
def test_zoh_gain_on_both_sides_of_the_switch(cuda, io, shape):
    """Exact ZOH with |Delta A| spread over about [5e-4, 0.3], so every call mixes
    the series branch (|Delta A| < 1/16) and the closed form."""
    n = SHAPES[shape].get("dstate", BASE.dstate)
    # |A| = 1 .. n: the step range that puts about half the (token, state) pairs
    # on each side of the switch
    lo, hi = (5e-4, 0.02) if n == 16 else (2e-3, 0.08)
    w = dataclasses.replace(BASE, io=io, name=f"zoh-switch-{shape}-{io}", dt_lo=lo, dt_hi=hi,
                            **SHAPES[shape])
    inp = synth.make_scan_inputs(w)
    inp["delta"] = (f64(inp["delta"]) * 0.1).astype(np.float32)
    inp["delta"] = torch.from_numpy(inp["delta"]).to(synth.io_dtype(io))
    dl = np.log1p(np.exp(f64(inp["delta"]) + f64(inp["delta_bias"])))
    a = np.abs(f64(inp["A"]))
    va = dl[..., None] * a[None, None]
    assert (va < 1 / 16).mean() > 0.2 and (va > 1 / 16).mean() > 0.2
    out, last, ref, ref_last, _ = scan_both(inp, cuda, zoh=True)
    tol = TOL[synth.io_dtype(io)]
    assert rel_err(f64(out), ref) <= tol
    assert rel_err(f64(last), ref_last) <= tol


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("n", [4, 16])
def test_decode_step_at_the_limits(cuda, io, zoh, n):
    """One ssm_state_update over tokens at Delta = 0, ordinary and Delta = 100
    (a third of the channels each): the held channels keep their state bit for
    bit, every output and state within the bound of the oracle's step."""
    w = dataclasses.replace(BASE, io=io, seqlen=1, dstate=n, name=f"decode-limits-{io}")
    inp = synth.make_scan_inputs(w)
    d = inp["delta"].clone()
    d[:, :, 0::3] = -1.0e4
    d[:, :, 2::3] = 100.0
    inp["delta"] = d
    inp["delta_bias"] = torch.zeros_like(inp["delta_bias"])
    dev = to_device(inp, cuda)
    state = dev["initial_state"].clone()
    out = ops.state_update(state, dev["x"][:, 0], dev["delta"][:, 0], dev["A"], dev["B"][:, 0],
                           dev["C"][:, 0], dev["D"], dev["z"][:, 0], dev["delta_bias"],
                           discretization="zoh" if zoh else "euler")
    torch.cuda.synchronize()
    ref, ref_last = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                                    f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                                    delta_bias=f64(inp["delta_bias"]),
                                    initial_state=f64(inp["initial_state"]), zoh=zoh)
    assert torch.equal(state[:, 0::3], dev["initial_state"][:, 0::3])
    tol = TOL[synth.io_dtype(io)]
    assert rel_err(f64(out), ref[:, 0]) <= tol
    assert rel_err(f64(state), ref_last) <= tol
