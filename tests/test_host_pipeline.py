"""GPU parity of ssm_scan_fwd_host (the scan of host-resident tensors,
pipelined over slices: whole sequences, or runs of steps of one sequence with
the state carried on the device) against the fp64 oracle, and against the
device-resident call; the forward's bounds (1e-4 fp32 I/O, 1e-2 bf16 I/O)."""
import dataclasses

import pytest
import torch

from parity import TOL, f64, oracle_full, rel_err
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu

BASE = synth.ScanWorkload("host-pipe", 5, 300, 72, 16, "bf16", 17, init_state=True)


def run_host(inp, cuda, slice_batch):
    pin = lambda t: None if t is None else t.pin_memory()
    out, last = ops.scan_fwd_host(pin(inp["x"]), pin(inp["delta"]), inp["A"].to(cuda), pin(inp["B"]),
                                  pin(inp["C"]), D=inp["D"].to(cuda), z=pin(inp["z"]),
                                  delta_bias=inp["delta_bias"].to(cuda),
                                  initial_state=pin(inp["initial_state"]), slice_batch=slice_batch)
    torch.cuda.synchronize()
    return out, last


@pytest.mark.parametrize("slice_batch", [0, 1, 2, 5, -64, -100, -299])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_host_pipeline(cuda, slice_batch, io):
    w = dataclasses.replace(BASE, io=io, seed=17 + abs(slice_batch))
    inp = synth.make_scan_inputs(w)
    out, last = run_host(inp, cuda, slice_batch)
    ref, ref_last = oracle_full(inp)
    tol = TOL[inp["x"].dtype]
    assert rel_err(f64(out), ref) <= tol and rel_err(f64(last), ref_last) <= tol


@pytest.mark.parametrize("slice_batch", [2, -128])
def test_host_pipeline_matches_device_call(cuda, slice_batch):
    inp = synth.make_scan_inputs(dataclasses.replace(BASE, with_z=False, init_state=False))
    out, last = run_host(inp, cuda, slice_batch)
    dev = {k: (None if v is None else v.to(cuda)) for k, v in inp.items()}
    dout, dlast = ops.scan_fwd(**dev)
    torch.cuda.synchronize()
    assert rel_err(f64(out), f64(dout)) <= 1e-2 and rel_err(f64(last), f64(dlast)) <= 1e-4


@pytest.mark.parametrize("slice_batch", [1, -1000, -2500])
def test_host_pipeline_long_sequences_chunked(cuda, slice_batch):
    """One sequence per slice, or runs of 1000 / 2500 steps of it: each slice
    takes the chunked (carry) plan, and the runs carry the state across."""
    w = synth.ScanWorkload("host-long", 3, 6000, 48, 16, "bf16", 27, dt_lo=1e-4, dt_hi=1e-2,
                           init_state=True)
    inp = synth.make_scan_inputs(w)
    out, last = run_host(inp, cuda, slice_batch)
    ref, ref_last = oracle_full(inp)
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]
    assert rel_err(f64(last), ref_last) <= TOL[torch.bfloat16]


def test_host_pipeline_full_size_sampled(cuda):
    """The Mamba-1.4B layer (4 x 8192 x 4096 x 16, bf16) from pinned host
    memory, as the benchmark's end-to-end figure runs it (runs of 2048 steps
    of one sequence, 16 slices): sampled channels of every sampled sequence (all 8192 tokens)
    and their final states against the oracle."""
    from parity import oracle_sampled, sample_channels
    w = synth.MAMBA_1P4B
    inp = synth.make_scan_inputs(w, device=str(cuda))
    host = {k: (None if v is None else v.cpu()) for k, v in inp.items()}
    out, last = run_host(host, cuda, 0)
    tol = TOL[inp["x"].dtype]
    for b, (ds, ref, ref_last) in oracle_sampled(inp, sample_channels(w.batch, w.dim)).items():
        idx = torch.tensor(ds)
        assert rel_err(f64(out[b].index_select(-1, idx)), ref) <= tol, (b, ds)
        assert rel_err(f64(last[b].index_select(0, idx)), ref_last) <= tol, (b, ds)


@pytest.mark.parametrize("with_state", [False, True])
def test_host_pipeline_runs_without_last_state(cuda, with_state):
    """Runs of 100 steps through the C ABI with no last_state requested: the
    state still passes from run to run on the device (and none is copied
    out), with and without an initial state."""
    w = dataclasses.replace(BASE, seed=71, init_state=with_state)
    inp = synth.make_scan_inputs(w)
    pin = lambda t: None if t is None else t.pin_memory()
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    need = binding.ssm_scan_fwd_host_workspace_size(desc, -100)
    wsb = torch.empty(need + 256, dtype=torch.uint8, device=cuda)
    ws = wsb[(256 - wsb.data_ptr() % 256) % 256:]
    out = torch.empty(inp["x"].shape, dtype=inp["x"].dtype).pin_memory()
    st = binding.ssm_scan_fwd_host(desc, -100, pin(inp["x"]), pin(inp["delta"]), inp["A"].to(cuda),
                                   pin(inp["B"]), pin(inp["C"]), inp["D"].to(cuda), pin(inp["z"]),
                                   inp["delta_bias"].to(cuda), out, None, pin(inp["initial_state"]), ws,
                                   ws.numel())
    torch.cuda.synchronize()
    assert st == binding.SSM_OK
    ref, _ = oracle_full(inp)
    assert rel_err(f64(out), ref) <= TOL[inp["x"].dtype]
