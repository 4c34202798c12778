"""GPU parity of ssm_state_update (decode) against the fp64 oracle's
recurrence, step by step, and decode == scan."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import ops, synth

pytestmark = pytest.mark.gpu

SMALL = synth.DecodeWorkload("decode-small", 3, 72, 16, 12, "bf16", 41)


def oracle_chain(inp, bsel, dsel, steps):
    """Oracle decode chain for channels dsel of sequences bsel; returns the
    per-step outputs (steps, nb, nd) and the states after each step."""
    idx = torch.tensor(dsel)
    bidx = torch.tensor(bsel)
    cpu = {k: v.cpu() for k, v in inp.items()}
    pick = lambda t: f64(t.index_select(-2, bidx).index_select(-1, idx))  # (..., nb, nd)
    st = f64(cpu["state"].index_select(0, bidx).index_select(1, idx))
    A = f64(cpu["A"].index_select(0, idx))
    D, bias = f64(cpu["D"].index_select(0, idx)), f64(cpu["delta_bias"].index_select(0, idx))
    outs, states = [], []
    for s in range(steps):
        o, st = oracle.state_update(st, pick(cpu["x"][s]), pick(cpu["delta"][s]), A,
                                    f64(cpu["B"][s].index_select(0, bidx)),
                                    f64(cpu["C"][s].index_select(0, bidx)), D, pick(cpu["z"][s]), bias)
        outs.append(o)
        states.append(st)
    return outs, states


def run_chain(inp, steps, check):
    state = inp["state"].clone()
    for s in range(steps):
        out = ops.state_update(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s],
                               inp["C"][s], inp["D"], inp["z"][s], inp["delta_bias"])
        check(s, out, state)
    return state


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_small_all_channels(cuda, n, io):
    w = dataclasses.replace(SMALL, dstate=n, io=io, seed=50 + n)
    inp = to_device(synth.make_decode_inputs(w), cuda)
    ref_out, ref_st = oracle_chain(inp, list(range(w.batch)), list(range(w.dim)), w.steps)
    tol = TOL[synth.io_dtype(io)]

    def check(s, out, state):
        torch.cuda.synchronize()
        assert rel_err(f64(out), ref_out[s]) <= tol, (s, rel_err(f64(out), ref_out[s]))
        assert rel_err(f64(state), ref_st[s]) <= tol
    run_chain(inp, w.steps, check)


def test_decode_full_size_128_steps(cuda):
    """256 sequences x 5120 channels x N=16, fp32 state ~ N(0,1) resident on the
    device, 128 chained steps; sampled channels checked at every step."""
    w = synth.DECODE
    inp = synth.make_decode_inputs(w, device=str(cuda))
    bsel, dsel = [0, 97, 255], [0, 1, 2560, 4095, 5119]
    ref_out, ref_st = oracle_chain(inp, bsel, dsel, w.steps)
    bi, di = torch.tensor(bsel, device=cuda), torch.tensor(dsel, device=cuda)
    tol = TOL[torch.bfloat16]
    worst = [0.0, 0.0]

    def check(s, out, state):
        got = f64(out.index_select(0, bi).index_select(1, di))
        e = rel_err(got, ref_out[s])
        worst[0] = max(worst[0], e)
        assert e <= tol, (s, e)
        if s % 32 == 31:
            gs = f64(state.index_select(0, bi).index_select(1, di))
            es = rel_err(gs, ref_st[s])
            worst[1] = max(worst[1], es)
            assert es <= tol, (s, es)
    final = run_chain(inp, w.steps, check)
    assert torch.isfinite(final).all()


def test_decode_equals_scan(cuda):
    """T decode steps from h0 equal one scan over the same T tokens."""
    T = 40
    w = synth.ScanWorkload("dec-vs-scan", 2, T, 72, 16, "f32", 61, init_state=True)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    out, last = ops.scan_fwd(**inp)
    state = inp["initial_state"].clone()
    outs = []
    for t in range(T):
        outs.append(ops.state_update(state, inp["x"][:, t].contiguous(), inp["delta"][:, t].contiguous(),
                                     inp["A"], inp["B"][:, t].contiguous(), inp["C"][:, t].contiguous(),
                                     inp["D"], inp["z"][:, t].contiguous(), inp["delta_bias"]))
    torch.cuda.synchronize()
    assert rel_err(f64(torch.stack(outs, 1)), f64(out)) <= 1e-4
    assert rel_err(f64(state), f64(last)) <= 1e-4


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_element_aligned_pointers(cuda, io):
    """A, B and C one element past a 16-byte boundary (element-aligned, which
    the contract accepts): the step takes element loads and matches the oracle."""
    w = dataclasses.replace(SMALL, io=io, steps=3, seed=77)
    inp = to_device(synth.make_decode_inputs(w), cuda)

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        return v

    A, Bs, Cs = shifted(inp["A"]), shifted(inp["B"]), shifted(inp["C"])
    assert A.data_ptr() % 16 != 0 and Bs.data_ptr() % 8 != 0
    ref_out, ref_st = oracle_chain(inp, list(range(w.batch)), list(range(w.dim)), w.steps)
    state = inp["state"].clone()
    tol = TOL[synth.io_dtype(io)]
    for s in range(w.steps):
        out = ops.state_update(state, inp["x"][s], inp["delta"][s], A, Bs[s], Cs[s], inp["D"],
                               inp["z"][s], inp["delta_bias"])
        torch.cuda.synchronize()
        assert rel_err(f64(out), ref_out[s]) <= tol
        assert rel_err(f64(state), ref_st[s]) <= tol
