"""ssm_scan_fwd_noalloc, the scan entry point for callers that cannot
allocate device memory (an operator plug-in handed only its input and output
buffers, or a latency-bound loop that must not call cudaMalloc).  It runs the
same kernels as ssm_scan_fwd with a caller workspace, so its results must be
bit-identical to that entry point's, call after call, although every call
reuses one fixed device scratch array; one case is also held against the
oracle.

This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests.
"""
import dataclasses

import pytest
import torch

from parity import TOL, f64, oracle_full, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu

# Few channels over a long sequence: the plan cuts time into chunks, so the
# scratch array is really used.
CHUNKED = synth.ScanWorkload("noalloc-chunked", 1, 6000, 48, 16, "bf16", 71,
                             dt_lo=1e-4, dt_hi=1e-2, init_state=True)


def noalloc_scan(inp):
    x = inp["x"]
    bsz, seqlen, dim = x.shape
    dstate = inp["A"].shape[1]
    out = torch.empty_like(x)
    last = torch.empty((bsz, dim, dstate), dtype=torch.float32, device=x.device)
    desc = binding.make_desc(bsz, seqlen, dim, dstate, x.dtype)
    st = binding.ssm_scan_fwd_noalloc(desc, x, inp["delta"], inp["A"], inp["B"], inp["C"],
                                      inp["D"], inp["z"], inp["delta_bias"], out, last,
                                      inp["initial_state"])
    assert st == binding.SSM_OK, binding.ssm_status_string(st)
    return out, last


def test_noalloc_matches_workspace_entry_point(cuda):
    cases = [CHUNKED,
             dataclasses.replace(CHUNKED, seed=72),                      # same shape, new data
             dataclasses.replace(CHUNKED, io="f32", dim=24, seqlen=5000, seed=73)]  # new layout
    for i, w in enumerate(cases):
        d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, synth.io_dtype(w.io))
        need = binding.ssm_scan_workspace_size(d)
        assert 0 < need <= binding.SSM_NOALLOC_SCRATCH_BYTES
        inp_cpu = synth.make_scan_inputs(w)
        inp = to_device(inp_cpu, cuda)
        ref_out, ref_last = ops.scan_fwd(**inp)          # caller-provided workspace
        out, last = noalloc_scan(inp)                     # fixed scratch, consecutive calls
        out2, last2 = noalloc_scan(inp)                   # the same call again: the scratch
        torch.cuda.synchronize()                          # holds the last call's carries
        # the same kernels on the same inputs: bit-identical results
        assert torch.equal(out, ref_out) and torch.equal(last, ref_last), w.name
        assert torch.equal(out2, out) and torch.equal(last2, last), w.name
        if i == 0:
            tol = TOL[synth.io_dtype(w.io)]
            ref, ref_state = oracle_full(inp_cpu)
            assert rel_err(f64(out), ref) <= tol
            assert rel_err(f64(last), ref_state) <= tol


def test_noalloc_rejects_problems_beyond_its_scratch(cuda):
    # dstate 64 over 2048 channels of a 262144-token sequence needs ~17 MB of carry scratch
    d = binding.make_desc(1, 262144, 2048, 64, torch.bfloat16)
    assert binding.ssm_scan_workspace_size(d) > binding.SSM_NOALLOC_SCRATCH_BYTES
    sentinel = torch.full((16,), 3.0, device=cuda)
    p = sentinel.data_ptr()
    st = binding.ssm_scan_fwd_noalloc(d, p, p, p, p, p, None, None, None, p, None, None)
    torch.cuda.synchronize()
    assert st == binding.SSM_ERR_UNSUPPORTED
    assert torch.all(sentinel == 3.0)
