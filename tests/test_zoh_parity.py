"""GPU parity of the exact zero-order-hold discretisation (ssm_scan_fwd_ex /
ssm_state_update_ex with SSM_DISC_ZOH) against the fp64 oracle's ZOH scan,
through the C ABI; the forward's elementwise bounds (1e-4 fp32 I/O, 1e-2
bf16 I/O, outputs and final state)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu


def check_zoh(w, cuda):
    inp = synth.make_scan_inputs(w)
    dev = to_device(inp, cuda)
    out, last = ops.scan_fwd(**dev, discretization="zoh")
    torch.cuda.synchronize()
    ref, ref_last = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                                    f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                                    delta_bias=f64(inp["delta_bias"]),
                                    initial_state=f64(inp["initial_state"]), zoh=True)
    tol = TOL[inp["x"].dtype]
    e_out, e_last = rel_err(f64(out), ref), rel_err(f64(last), ref_last)
    assert e_out <= tol, f"{w.name}: out error {e_out:.3e}"
    assert e_last <= tol, f"{w.name}: last_state error {e_last:.3e}"
    # the variant must actually differ from the first-order form
    eul, _ = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                             f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                             delta_bias=f64(inp["delta_bias"]),
                             initial_state=f64(inp["initial_state"]))
    return e_out, rel_err(eul, ref)


SMALL = synth.ScanWorkload("zoh-small", 2, 300, 72, 16, "bf16", 31, init_state=True,
                           dt_lo=0.02, dt_hi=0.5)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_warp_specialised(cuda, io):
    e, gap = check_zoh(dataclasses.replace(SMALL, io=io, name=f"zoh-{io}"), cuda)
    assert gap > 10 * TOL[synth.io_dtype(io)], "inputs too mild to tell ZOH from first order"


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_small_steps_series_branch(cuda, io):
    """Delta A below 1/16 everywhere: the series branch of the gain."""
    check_zoh(dataclasses.replace(SMALL, io=io, dt_lo=1e-4, dt_hi=2e-3, name=f"zoh-small-dt-{io}"),
              cuda)


@pytest.mark.parametrize("n", [1, 4, 8, 32, 64])
def test_zoh_general_kernel(cuda, n):
    check_zoh(dataclasses.replace(SMALL, io="f32", dstate=n, seed=60 + n, name=f"zoh-n{n}"), cuda)


def test_zoh_random_A(cuda):
    check_zoh(dataclasses.replace(SMALL, io="f32", random_A=True, name="zoh-randA"), cuda)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_chunked_long_sequence(cuda, io):
    w = synth.ScanWorkload(f"zoh-chunked-{io}", 1, 6000, 48, 16, io, 23, dt_lo=1e-4, dt_hi=1e-2,
                           init_state=True)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, synth.io_dtype(io))
    assert binding.ssm_scan_plan(d).nchunk > 1
    check_zoh(w, cuda)


@pytest.mark.parametrize("L", [1, 17, 33])
def test_zoh_edge_lengths(cuda, L):
    check_zoh(dataclasses.replace(SMALL, seqlen=L, seed=70 + L, name=f"zoh-L{L}"), cuda)


@pytest.mark.parametrize("n", [4, 16])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_decode_chain(cuda, n, io):
    """Decode steps with ZOH against the oracle's ZOH scan one token at a
    time (initial state = the previous state)."""
    w = synth.DecodeWorkload("zoh-decode", 3, 72, n, 6, io, 90 + n, dt_lo=0.02, dt_hi=0.5)
    inp = synth.make_decode_inputs(w)
    dev = to_device(inp, cuda)
    state = dev["state"].clone()
    ref_state = f64(inp["state"])
    tol = TOL[synth.io_dtype(io)]
    for s in range(w.steps):
        out = ops.state_update(state, dev["x"][s], dev["delta"][s], dev["A"], dev["B"][s],
                               dev["C"][s], dev["D"], dev["z"][s], dev["delta_bias"],
                               discretization="zoh")
        torch.cuda.synchronize()
        tok = lambda t: f64(t[s])[:, None, :]
        ref, ref_state = oracle.scan_fwd(tok(inp["x"]), tok(inp["delta"]), f64(inp["A"]),
                                         tok(inp["B"]), tok(inp["C"]), D=f64(inp["D"]),
                                         z=tok(inp["z"]), delta_bias=f64(inp["delta_bias"]),
                                         initial_state=ref_state, zoh=True)
        assert rel_err(f64(out), ref[:, 0, :]) <= tol, s
        assert rel_err(f64(state), ref_state) <= tol, s


def test_euler_option_equals_plain_call(cuda):
    """SSM_DISC_EULER through the _ex call is the plain scan, bit for bit."""
    inp = to_device(synth.make_scan_inputs(SMALL), cuda)
    a, la = ops.scan_fwd(**inp)
    desc = binding.make_desc(SMALL.batch, SMALL.seqlen, SMALL.dim, SMALL.dstate, inp["x"].dtype)
    out = torch.empty_like(inp["x"])
    last = torch.empty_like(la)
    need = binding.ssm_scan_workspace_size(desc)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=cuda)
    st = binding.ssm_scan_fwd_ex(desc, binding.make_opts("euler"), inp["x"], inp["delta"], inp["A"],
                                 inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"], out,
                                 last, inp["initial_state"], ws, ws.numel())
    torch.cuda.synchronize()
    assert st == binding.SSM_OK and torch.equal(out, a) and torch.equal(last, la)


def test_zoh_full_size_sampled(cuda):
    """The Mamba-1.4B layer (4 x 8192 x 4096 x 16, bf16) with exact ZOH, as the
    benchmark times it: every output of sampled channels and their final
    states against the oracle's ZOH scan on those channels alone."""
    from parity import sample_channels
    w = synth.MAMBA_1P4B
    inp = synth.make_scan_inputs(w, device=str(cuda))
    out, last = ops.scan_fwd(**inp, discretization="zoh")
    torch.cuda.synchronize()
    tol = TOL[inp["x"].dtype]
    for b, ds in sample_channels(w.batch, w.dim):
        idx = torch.tensor(ds, device=cuda)
        tok = lambda t: f64(t[b].index_select(-1, idx))[None]
        par = lambda t: f64(t.index_select(0, idx))
        ref, ref_last = oracle.scan_fwd(tok(inp["x"]), tok(inp["delta"]), par(inp["A"]),
                                        f64(inp["B"][b])[None], f64(inp["C"][b])[None],
                                        D=par(inp["D"]), z=tok(inp["z"]),
                                        delta_bias=par(inp["delta_bias"]), zoh=True)
        assert rel_err(tok(out), ref) <= tol, (b, ds, rel_err(tok(out), ref))
        assert rel_err(f64(last[b].index_select(0, idx))[None], ref_last) <= tol, (b, ds)
