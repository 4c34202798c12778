"""GPU parity of the selection projections (ssm_selection_proj_fwd: x_proj
split into dt_low, B, C; dt_proj) on the tensor cores against the oracle's
fp64 matmuls, through the C ABI.

Bound: elementwise |y - y_ref| <= 1e-2 (1 + |y_ref|) for every output -- the
bf16 I/O bound: the GPU rounds each output to bf16 once (2^-9 relative) and
feeds the bf16-rounded dt_low into dt_proj, a relative perturbation of 2^-9
per term of an fp32 sum whose magnitude the (1 + |ref|) form covers."""
import numpy as np
import pytest
import torch

import oracle
from parity import f64, rel_err
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu
TOL = 1e-2


def check_proj(bsz, L, dim, R, N, seed, cuda):
    inp = synth.make_proj_inputs(bsz, L, dim, R, N, seed)
    dev = {k: v.to(cuda) for k, v in inp.items()}
    dt_low, Bm, Cm, delta = ops.selection_proj(dev["x"], dev["W_x"], dev["W_dt"], R, N)
    torch.cuda.synchronize()
    ref = oracle.selection_proj(f64(inp["x"]), f64(inp["W_x"]), f64(inp["W_dt"]), R)
    errs = [rel_err(f64(g), r) for g, r in zip((dt_low, Bm, Cm, delta), ref)]
    for name, e in zip(("dt_low", "B", "C", "delta"), errs):
        assert e <= TOL, f"({bsz},{L},{dim},R={R},N={N}) {name}: {e:.3e}"
    return errs


def test_proj_mamba_like_small(cuda):
    check_proj(2, 300, 512, 32, 16, 1, cuda)


@pytest.mark.parametrize("shape", [(1, 128, 64, 16, 8), (1, 1, 64, 8, 4), (3, 77, 256, 48, 16),
                                   (2, 200, 1024, 64, 16), (1, 130, 320, 128, 16),
                                   (1, 64, 96, 200, 8)])
def test_proj_shapes(cuda, shape):
    """Ragged token counts (partial 128-row tiles), K not a multiple of 64,
    every x_proj tile width up to 256."""
    check_proj(*shape, seed=sum(shape), cuda=cuda)


def test_proj_mamba_1p4b_rows_sampled(cuda):
    """Mamba-1.4B shapes (4 x 8192 tokens, dim 4096, R 128, N 16): sampled
    token rows against the oracle run on those rows alone."""
    bsz, L, dim, R, N = 4, 8192, 4096, 128, 16
    inp = synth.make_proj_inputs(bsz, L, dim, R, N, 7, device=str(cuda))
    dt_low, Bm, Cm, delta = ops.selection_proj(inp["x"], inp["W_x"], inp["W_dt"], R, N)
    torch.cuda.synchronize()
    rows = [(0, 0), (0, 8191), (1, 4096), (3, 127), (3, 128), (2, 5000)]
    x = torch.stack([inp["x"][b, t] for b, t in rows])[None]
    ref = oracle.selection_proj(f64(x), f64(inp["W_x"]), f64(inp["W_dt"]), R)
    got = [torch.stack([t[b, l] for b, l in rows])[None] for t in (dt_low, Bm, Cm, delta)]
    for name, g, r in zip(("dt_low", "B", "C", "delta"), got, ref):
        assert rel_err(f64(g), r) <= TOL, name


def test_proj_feeds_the_scan(cuda):
    """delta_raw, B, C from the projections go straight into ssm_scan_fwd.
    Each stage is held to the bf16 bound against the oracle on that stage's
    own inputs: the projections against the oracle's projections, and the
    scan against the oracle's scan fed the very bf16 values the GPU scan
    consumed (the bf16 rounding of the projection outputs is an input to the
    scan, not an error of it)."""
    bsz, L, dim, R, N = 2, 256, 256, 32, 16
    p = synth.make_proj_inputs(bsz, L, dim, R, N, 11)
    s = synth.make_scan_inputs(synth.ScanWorkload("proj-scan", bsz, L, dim, N, "bf16", 12))
    dev = {k: v.to(cuda) for k, v in p.items()}
    _, Bm, Cm, delta = ops.selection_proj(dev["x"], dev["W_x"], dev["W_dt"], R, N)
    out, last = ops.scan_fwd(dev["x"], delta, s["A"].to(cuda), Bm, Cm, D=s["D"].to(cuda),
                             z=s["z"].to(cuda), delta_bias=s["delta_bias"].to(cuda))
    torch.cuda.synchronize()
    _, rB, rC, rdelta = oracle.selection_proj(f64(p["x"]), f64(p["W_x"]), f64(p["W_dt"]), R)
    for name, g, r in (("B", Bm, rB), ("C", Cm, rC), ("delta", delta, rdelta)):
        assert rel_err(f64(g), r) <= TOL, name
    ref, ref_last = oracle.scan_fwd(f64(p["x"]), f64(delta), f64(s["A"]), f64(Bm), f64(Cm),
                                    D=f64(s["D"]), z=f64(s["z"]), delta_bias=f64(s["delta_bias"]))
    assert rel_err(f64(out), ref) <= TOL
    assert rel_err(f64(last), ref_last) <= TOL


def test_proj_rejections(cuda):
    d = binding.make_desc(1, 16, 60, 16, torch.bfloat16)      # dim not a multiple of 8
    x = torch.zeros(1, 16, 64, dtype=torch.bfloat16, device=cuda)
    assert binding.ssm_selection_proj_fwd(d, binding.ssm_proj_desc(16, 0), x, x, x, None, x, x, x,
                                          None) == binding.SSM_ERR_UNSUPPORTED
    d = binding.make_desc(1, 16, 64, 128, torch.bfloat16)     # R + 2N > 256
    assert binding.ssm_selection_proj_fwd(d, binding.ssm_proj_desc(16, 0), x, x, x, None, x, x, x,
                                          None) == binding.SSM_ERR_UNSUPPORTED
    d = binding.make_desc(1, 16, 64, 16, torch.float32)       # fp32 I/O
    assert binding.ssm_selection_proj_fwd(d, binding.ssm_proj_desc(16, 0), x, x, x, None, x, x, x,
                                          None) == binding.SSM_ERR_UNSUPPORTED


def test_proj_epilogue_finishes_delta(cuda):
    """Bias and softplus in dt_proj's epilogue: delta is the step itself, and
    the scan runs without softplus or bias; against the oracle's raw
    projection followed by the oracle's scan with softplus and bias."""
    bsz, L, dim, R, N = 2, 256, 256, 32, 16
    p = synth.make_proj_inputs(bsz, L, dim, R, N, 21)
    s = synth.make_scan_inputs(synth.ScanWorkload("proj-sp", bsz, L, dim, N, "bf16", 22))
    dev = {k: v.to(cuda) for k, v in p.items()}
    bias = s["delta_bias"].to(cuda)
    _, Bm, Cm, dt = ops.selection_proj(dev["x"], dev["W_x"], dev["W_dt"], R, N, delta_bias=bias,
                                       delta_softplus=True)
    out, last = ops.scan_fwd(dev["x"], dt, s["A"].to(cuda), Bm, Cm, D=s["D"].to(cuda),
                             z=s["z"].to(cuda), delta_softplus=False)
    torch.cuda.synchronize()
    _, rB, rC, rdelta = oracle.selection_proj(f64(p["x"]), f64(p["W_x"]), f64(p["W_dt"]), R)
    sp = np.logaddexp(0.0, rdelta + f64(s["delta_bias"]))
    assert rel_err(f64(dt), sp) <= TOL
    # the scan against the oracle's scan of the step the epilogue produced
    ref, ref_last = oracle.scan_fwd(f64(p["x"]), f64(dt), f64(s["A"]), f64(Bm), f64(Cm),
                                    D=f64(s["D"]), z=f64(s["z"]), delta_softplus=False)
    assert rel_err(f64(out), ref) <= TOL
    assert rel_err(f64(last), ref_last) <= TOL
