"""GPU parity of the scan with dt_proj fused in front (ssm_proj_scan_fwd),
through the C ABI, against the fp64 oracle: the oracle's second selection
projection (delta_raw = dt_low W_dt^T) followed by the oracle's scan, fed the
same bf16 dt_low, B and C the GPU consumed ("Mamba的三大创新", the selection
mechanism: Delta computed from the input).

Bound: the forward's bf16 bound, elementwise |y - y_ref| <= 1e-2 (1 + |y_ref|)
for the output and the final state.  The fused kernel forms the raw step in
fp32 from the bf16 operands (no bf16 rounding of delta_raw, unlike the
unfused pipeline), so it sits closer to the oracle than the unfused path."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, sample_channels
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu


def make_case(bsz, L, dim, R, seed, cuda, init_state=False, dt=(1e-3, 1e-1)):
    """dt_low, B, C from the GPU's x_proj on synthetic x and weights; A, D,
    z, the bias (and h0) from the scan recipe."""
    p = synth.make_proj_inputs(bsz, L, dim, R, 16, seed)
    w = synth.ScanWorkload("proj-scan", bsz, L, dim, 16, "bf16", seed + 1, init_state=init_state,
                           dt_lo=dt[0], dt_hi=dt[1])
    s = synth.make_scan_inputs(w)
    dev = {k: v.to(cuda) for k, v in p.items()}
    dt_low, Bm, Cm, _ = ops.selection_proj(dev["x"], dev["W_x"], dev["W_dt"], R, 16)
    sd = {k: (None if v is None else v.to(cuda)) for k, v in s.items()}
    return dict(x=dev["x"], dt_low=dt_low, W_dt=dev["W_dt"], A=sd["A"], B=Bm, C=Cm, D=sd["D"],
                z=sd["z"], delta_bias=sd["delta_bias"], initial_state=sd["initial_state"]), dev["W_x"]


def oracle_of(c):
    draw = oracle.dt_proj(f64(c["dt_low"]), f64(c["W_dt"]))
    return oracle.scan_fwd(f64(c["x"]), draw, f64(c["A"]), f64(c["B"]), f64(c["C"]), D=f64(c["D"]),
                           z=f64(c["z"]), delta_bias=f64(c["delta_bias"]),
                           initial_state=f64(c["initial_state"]))


@pytest.mark.parametrize("R", [64, 128])
@pytest.mark.parametrize("shape", [(2, 256, 256), (1, 300, 40), (3, 33, 64)])
def test_fused_against_oracle(cuda, R, shape):
    """Whole tiles, a partial last tile (300 = 18 x 16 + 12 steps, 33 steps),
    and 40 channels: a partial channel block (W_dt rows past the end read as 0)."""
    c, _ = make_case(*shape, R, seed=5 + R + shape[1], cuda=cuda, init_state=True)
    out, last = ops.proj_scan_fwd(**c)
    torch.cuda.synchronize()
    ref, ref_last = oracle_of(c)
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]
    assert rel_err(f64(last), ref_last) <= TOL[torch.bfloat16]


def test_fused_equals_unfused_pipeline(cuda):
    """The fused path and the unfused one (dt_proj's bf16 delta_raw, then
    ssm_scan_fwd) agree within the bf16 bound; they differ only by the bf16
    rounding of the raw step."""
    c, W_x = make_case(2, 512, 512, 128, 77, cuda)
    out, last = ops.proj_scan_fwd(**c)
    _, _, _, draw = ops.selection_proj(c["x"], W_x, c["W_dt"], 128, 16)   # bf16 delta_raw
    out2, last2 = ops.scan_fwd(c["x"], draw, c["A"], c["B"], c["C"], D=c["D"], z=c["z"],
                               delta_bias=c["delta_bias"])
    torch.cuda.synchronize()
    assert rel_err(f64(out), f64(out2)) <= TOL[torch.bfloat16]
    assert rel_err(f64(last), f64(last2)) <= TOL[torch.bfloat16]


def test_fused_chunked_long_sequence(cuda):
    """Few channels over a long sequence: the time axis is cut into chunks,
    so the fused aggregate pass and the carry run too."""
    c, _ = make_case(1, 6000, 48, 64, 91, cuda, init_state=True, dt=(1e-4, 1e-2))
    d = binding.make_desc(1, 6000, 48, 16, torch.bfloat16)
    assert binding.ssm_scan_plan(d).nchunk > 1
    out, last = ops.proj_scan_fwd(**c)
    torch.cuda.synchronize()
    ref, ref_last = oracle_of(c)
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]
    assert rel_err(f64(last), ref_last) <= TOL[torch.bfloat16]


def test_fused_mamba_1p4b_layer_sampled(cuda):
    """The Mamba-1.4B layer (4 x 8192 tokens, dim 4096, R 128): sampled
    channels of every sequence against the oracle run on those channels."""
    bsz, L, dim, R = 4, 8192, 4096, 128
    c, _ = make_case(bsz, L, dim, R, 123, cuda)
    out, last = ops.proj_scan_fwd(**c)
    torch.cuda.synchronize()
    for b, ds in sample_channels(bsz, dim, per_batch=5, seed=3):
        idx = torch.tensor(ds, device=cuda)
        draw = oracle.dt_proj(f64(c["dt_low"][b])[None], f64(c["W_dt"].index_select(0, idx)))
        g = lambda t: f64(t[b].index_select(-1, idx))[None]
        vec = lambda t: f64(t.index_select(0, idx))
        ref, ref_last = oracle.scan_fwd(g(c["x"]), draw, f64(c["A"].index_select(0, idx)),
                                        f64(c["B"][b])[None], f64(c["C"][b])[None], D=vec(c["D"]),
                                        z=g(c["z"]), delta_bias=vec(c["delta_bias"]))
        assert rel_err(f64(out[b].index_select(-1, idx)), ref[0]) <= TOL[torch.bfloat16], (b, ds)
        assert rel_err(f64(last[b].index_select(0, idx)), ref_last[0]) <= TOL[torch.bfloat16]


def test_fused_rejections(cuda):
    c, _ = make_case(1, 64, 64, 64, 1, cuda)
    ws = torch.empty(16, dtype=torch.uint8, device=cuda)

    def call(desc, R):
        return binding.ssm_proj_scan_fwd(desc, binding.ssm_proj_desc(R, 0), c["x"], c["dt_low"],
                                         c["W_dt"], c["A"], c["B"], c["C"], c["D"], c["z"],
                                         c["delta_bias"], c["x"], None, None, ws, ws.numel())
    bf = torch.bfloat16
    assert call(binding.make_desc(1, 64, 64, 16, bf, True), 48) == binding.SSM_ERR_UNSUPPORTED
    assert call(binding.make_desc(1, 64, 64, 8, bf, True), 64) == binding.SSM_ERR_UNSUPPORTED
    assert call(binding.make_desc(1, 64, 64, 16, torch.float32, True), 64) == binding.SSM_ERR_UNSUPPORTED
    assert call(binding.make_desc(1, 64, 64, 16, bf, False), 64) == binding.SSM_ERR_UNSUPPORTED
    assert binding.ssm_proj_scan_fwd(binding.make_desc(1, 64, 64, 16, bf, True),
                                     binding.ssm_proj_desc(64, 1), c["x"], c["dt_low"], c["W_dt"],
                                     c["A"], c["B"], c["C"], None, None, None, c["x"], None, None,
                                     ws, ws.numel()) == binding.SSM_ERR_INVALID_ARG
