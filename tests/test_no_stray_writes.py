"""No kernel writes outside the tensors it is given: every output of the
backward, the decode step, the standalone conv, the LTI convolution, the
selection projections, the fused conv + scan and dt_proj + scan, and the
training forward's checkpoints lives at the start of a
larger buffer filled with a sentinel, and the tail must come back unchanged.
Shapes with a partial last tile of steps and a partial last block of
channels (the TMA stores clip there, the register paths mask), and the
outputs themselves checked against the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu

SENT = -77.0
PAD = 4096


def guarded(shape, dtype, device):
    """A tensor of `shape` at the start of a buffer PAD elements longer, all
    set to the sentinel; returns (view, tail)."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + PAD,), SENT, dtype=dtype, device=device)
    return buf[:n].view(shape), buf[n:]


def untouched(tail):
    return bool(torch.all(tail == SENT))


@pytest.mark.parametrize("dim,seqlen,io", [(40, 97, "bf16"), (48, 97, "f32"), (16, 33, "bf16")])
@pytest.mark.parametrize("ckpt", [False, True])
def test_bwd_writes_only_its_outputs(cuda, dim, seqlen, io, ckpt):
    """All nine gradients of ssm_scan_bwd_ex, with the states recomputed or
    read from the training forward's checkpoints."""
    w = synth.ScanWorkload(f"bwd-guard-{dim}-{seqlen}-{io}", 2, seqlen, dim, 16, io, 60 + dim,
                           init_state=True)
    inp = synth.make_scan_inputs(w)
    g = torch.Generator().manual_seed(7)
    dout = torch.randn(inp["x"].shape, generator=g).to(inp["x"].dtype)
    dl = torch.randn((w.batch, w.dim, w.dstate), generator=g)
    dev = to_device(inp, cuda)
    dt = inp["x"].dtype
    tok, st = tuple(inp["x"].shape), (w.batch, w.dim, w.dstate)
    f32 = torch.float32
    dx, tx = guarded(tok, dt, cuda)
    ddl, tdl = guarded(tok, dt, cuda)
    dz, tz = guarded(tok, dt, cuda)
    dA, tA = guarded((w.dim, w.dstate), f32, cuda)
    dB, tB = guarded((w.batch, w.seqlen, w.dstate), f32, cuda)
    dC, tC = guarded((w.batch, w.seqlen, w.dstate), f32, cuda)
    dD, tD = guarded((w.dim,), f32, cuda)
    db, tb = guarded((w.dim,), f32, cuda)
    di, ti = guarded(st, f32, cuda)
    ck = None
    if ckpt:
        ck = ops.checkpoint_buffer(dev["x"], dev["A"])
        ops.scan_fwd(**dev, checkpoints=ck)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, dt)
    need = binding.ssm_scan_bwd_ex_workspace_size(desc, ck is not None)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=cuda)
    status = binding.ssm_scan_bwd_ex(desc, dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                     dev["z"], dev["delta_bias"], dev["initial_state"], dout.to(cuda),
                                     dl.to(cuda), ck, dx, ddl, dA, dB, dC, dD, dz, db, di, ws, ws.numel())
    torch.cuda.synchronize()
    assert status == binding.SSM_OK
    for name, tail in (("dx", tx), ("ddelta", tdl), ("dz", tz), ("dA", tA), ("dB", tB), ("dC", tC),
                       ("dD", tD), ("ddelta_bias", tb), ("dinitial_state", ti)):
        assert untouched(tail), name
    ref = oracle.scan_bwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]), f64(inp["C"]),
                          f64(dout), D=f64(inp["D"]), z=f64(inp["z"]), delta_bias=f64(inp["delta_bias"]),
                          initial_state=f64(inp["initial_state"]), dlast_state=f64(dl))
    tol = TOL[dt]
    assert rel_err(f64(dx), ref["dx"]) <= tol
    assert rel_err(f64(ddl), ref["ddelta"]) <= tol
    assert rel_err(f64(dz), ref["dz"]) <= tol


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_writes_only_its_outputs(cuda, io):
    w = synth.ScanWorkload(f"decode-guard-{io}", 3, 1, 40, 16, io, 12, init_state=True)
    inp = synth.make_scan_inputs(w)
    dev = to_device(inp, cuda)
    state, ts = guarded((w.batch, w.dim, w.dstate), torch.float32, cuda)
    state.copy_(dev["initial_state"])
    out, to = guarded((w.batch, w.dim), inp["x"].dtype, cuda)
    ops.state_update(state, dev["x"][:, 0], dev["delta"][:, 0], dev["A"], dev["B"][:, 0], dev["C"][:, 0],
                     dev["D"], dev["z"][:, 0], dev["delta_bias"], out=out)
    torch.cuda.synchronize()
    assert untouched(ts) and untouched(to)
    ref, ref_last = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                                    f64(inp["C"]), D=f64(inp["D"]), z=f64(inp["z"]),
                                    delta_bias=f64(inp["delta_bias"]),
                                    initial_state=f64(inp["initial_state"]))
    tol = TOL[inp["x"].dtype]
    assert rel_err(f64(out), ref[:, 0]) <= tol
    assert rel_err(f64(state), ref_last) <= tol


@pytest.mark.parametrize("io,dim", [("bf16", 40), ("bf16", 64), ("f32", 36)])
def test_conv1d_writes_only_its_outputs(cuda, io, dim):
    """The standalone causal conv: output and the carried history."""
    w = synth.ScanWorkload(f"conv-guard-{io}-{dim}", 2, 97, dim, 16, io, 13)
    inp = synth.make_scan_inputs(w)
    width = 4
    g = torch.Generator().manual_seed(3)
    cw = torch.randn((dim, width), generator=g) * 0.5
    cb = torch.randn((dim,), generator=g) * 0.1
    hist = torch.randn((w.batch, dim, width - 1), generator=g)
    x = inp["x"].to(cuda)
    out, to = guarded(tuple(x.shape), x.dtype, cuda)
    st, tst = guarded((w.batch, dim, width - 1), torch.float32, cuda)
    got, got_state = ops.conv1d_fwd(x, cw.to(cuda), bias=cb.to(cuda), conv_state=hist.to(cuda), out=out,
                                    conv_state_out=st)
    torch.cuda.synchronize()
    assert untouched(to) and untouched(tst)
    ref, ref_state = oracle.conv1d_fwd(f64(inp["x"]), f64(cw), bias=f64(cb), conv_state=f64(hist), activation=True)
    assert rel_err(f64(got), ref) <= TOL[x.dtype]
    assert rel_err(f64(got_state), ref_state) <= 1e-6


@pytest.mark.parametrize("io,shape", [("bf16", (2, 300, 72)), ("bf16", (9, 129, 16)), ("f32", (2, 300, 72)),
                                      ("bf16", (1, 97, 33))])
def test_lti_conv_writes_only_its_outputs(cuda, io, shape):
    """The LTI convolution: bf16 with dim a multiple of 8 runs the tensor-core
    kernel, whose TMA stores clip at a partial block of 8 sequences and a
    partial group of 128 steps; the other two shapes run the CUDA-core kernel."""
    bsz, L, dim = shape
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[io]
    g = torch.Generator().manual_seed(L * dim)
    K = torch.randn((dim, L), generator=g) * torch.exp(-0.05 * torch.arange(L))[None, :]
    x = torch.randn((bsz, L, dim), generator=g).to(dt)
    z = torch.randn((bsz, L, dim), generator=g).to(dt)
    D = torch.randn(dim, generator=g)
    out, tail = guarded((bsz, L, dim), dt, cuda)
    got = ops.lti_conv_fwd(K.to(cuda), x.to(cuda), D=D.to(cuda), z=z.to(cuda), out=out)
    torch.cuda.synchronize()
    assert got.data_ptr() == out.data_ptr()
    assert untouched(tail)
    ref = oracle.lti_conv(f64(K), f64(x), D=f64(D), z=f64(z))
    assert rel_err(f64(out), ref) <= TOL[dt]


@pytest.mark.parametrize("shape", [(2, 97, 256, 32, 16), (3, 77, 320, 128, 16)])
def test_selection_proj_writes_only_its_outputs(cuda, shape):
    """x_proj's three outputs and dt_proj's delta, with a partial last tile of
    128 token rows (194 and 231 tokens)."""
    bsz, L, dim, R, N = shape
    inp = synth.make_proj_inputs(bsz, L, dim, R, N, sum(shape))
    dev = {k: v.to(cuda) for k, v in inp.items()}
    bf = torch.bfloat16
    dt_low, t1 = guarded((bsz, L, R), bf, cuda)
    Bm, t2 = guarded((bsz, L, N), bf, cuda)
    Cm, t3 = guarded((bsz, L, N), bf, cuda)
    delta, t4 = guarded((bsz, L, dim), bf, cuda)
    desc = binding.make_desc(bsz, L, dim, N, bf, False)
    st = binding.ssm_selection_proj_fwd(desc, binding.ssm_proj_desc(R, 0), dev["x"], dev["W_x"], dev["W_dt"],
                                        None, dt_low, Bm, Cm, delta)
    torch.cuda.synchronize()
    assert st == binding.SSM_OK
    for name, tail in (("dt_low", t1), ("B", t2), ("C", t3), ("delta", t4)):
        assert untouched(tail), name
    ref = oracle.selection_proj(f64(inp["x"]), f64(inp["W_x"]), f64(inp["W_dt"]), R)
    for name, g, r in zip(("dt_low", "B", "C", "delta"), (dt_low, Bm, Cm, delta), ref):
        assert rel_err(f64(g), r) <= 1e-2, name


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_scan_writes_only_its_outputs(cuda, io):
    """The fused conv + scan: output, final state and the carried conv history."""
    w = synth.ScanWorkload(f"convscan-guard-{io}", 2, 97, 40, 16, io, 31, init_state=True)
    inp = synth.make_scan_inputs(w)
    conv = synth.make_conv_inputs(w.batch, w.dim, 4, seed=32, with_bias=True, with_state=True)
    dev, cd = to_device(inp, cuda), to_device(conv, cuda)
    out, to = guarded(tuple(inp["x"].shape), inp["x"].dtype, cuda)
    last, tl = guarded((w.batch, w.dim, w.dstate), torch.float32, cuda)
    cst, tc = guarded((w.batch, w.dim, 3), torch.float32, cuda)
    ops.conv_scan_fwd(dev["x"], cd["conv_w"], dev["delta"], dev["A"], dev["B"], dev["C"], D=dev["D"],
                      z=dev["z"], delta_bias=dev["delta_bias"], conv_bias=cd["conv_bias"],
                      conv_state=cd["conv_state"], initial_state=dev["initial_state"], out=out,
                      last_state=last, conv_state_out=cst)
    torch.cuda.synchronize()
    assert untouched(to) and untouched(tl) and untouched(tc)
    xc, ref_cst = oracle.conv1d_fwd(f64(inp["x"]), f64(conv["conv_w"]), f64(conv["conv_bias"]),
                                    f64(conv["conv_state"]), True)
    ref, ref_last = oracle.scan_fwd(xc, f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]), f64(inp["C"]),
                                    D=f64(inp["D"]), z=f64(inp["z"]), delta_bias=f64(inp["delta_bias"]),
                                    initial_state=f64(inp["initial_state"]))
    tol = TOL[inp["x"].dtype]
    assert rel_err(f64(out), ref) <= tol
    assert rel_err(f64(last), ref_last) <= tol
    assert np.array_equal(f64(cst), ref_cst)


def test_proj_scan_writes_only_its_outputs(cuda):
    """The scan with dt_proj fused in front: 40 channels (a partial block of
    16) and 300 steps (a partial last tile)."""
    bsz, L, dim, R = 2, 300, 40, 64
    p = synth.make_proj_inputs(bsz, L, dim, R, 16, 41)
    s = synth.make_scan_inputs(synth.ScanWorkload("projscan-guard", bsz, L, dim, 16, "bf16", 42,
                                                  init_state=True))
    dev = {k: v.to(cuda) for k, v in p.items()}
    dt_low, Bm, Cm, _ = ops.selection_proj(dev["x"], dev["W_x"], dev["W_dt"], R, 16)
    sd = {k: (None if v is None else v.to(cuda)) for k, v in s.items()}
    out, to = guarded((bsz, L, dim), torch.bfloat16, cuda)
    last, tl = guarded((bsz, dim, 16), torch.float32, cuda)
    ops.proj_scan_fwd(dev["x"], dt_low, dev["W_dt"], sd["A"], Bm, Cm, D=sd["D"], z=sd["z"],
                      delta_bias=sd["delta_bias"], initial_state=sd["initial_state"], out=out, last_state=last)
    torch.cuda.synchronize()
    assert untouched(to) and untouched(tl)
    draw = oracle.dt_proj(f64(dt_low), f64(dev["W_dt"]))
    ref, ref_last = oracle.scan_fwd(f64(dev["x"]), draw, f64(sd["A"]), f64(Bm), f64(Cm), D=f64(sd["D"]),
                                    z=f64(sd["z"]), delta_bias=f64(sd["delta_bias"]),
                                    initial_state=f64(sd["initial_state"]))
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]
    assert rel_err(f64(last), ref_last) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dim,seqlen,io", [(40, 97, "bf16"), (48, 130, "f32")])
def test_checkpoints_write_only_their_buffer(cuda, dim, seqlen, io):
    """The training forward writes no further than ssm_scan_checkpoint_size
    bytes of checkpoints, and its output is the plain forward's."""
    w = synth.ScanWorkload(f"ckpt-guard-{dim}-{io}", 2, seqlen, dim, 16, io, 50 + dim, init_state=True)
    inp = synth.make_scan_inputs(w)
    dev = to_device(inp, cuda)
    n = binding.ssm_scan_checkpoint_size(binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate,
                                                           inp["x"].dtype)) // 4
    ck, tck = guarded((n,), torch.float32, cuda)
    out, _ = ops.scan_fwd(**dev, checkpoints=ck)
    torch.cuda.synchronize()
    assert untouched(tck)
    ref, _ = oracle.scan_fwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]), f64(inp["C"]),
                             D=f64(inp["D"]), z=f64(inp["z"]), delta_bias=f64(inp["delta_bias"]),
                             initial_state=f64(inp["initial_state"]))
    assert rel_err(f64(out), ref) <= TOL[inp["x"].dtype]
