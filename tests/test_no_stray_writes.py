"""No kernel writes outside the tensors it is given: every output of the
backward, the decode step and the standalone conv lives at the start of a
larger buffer filled with a sentinel, and the tail must come back unchanged.
Shapes with a partial last tile of steps and a partial last block of
channels (the TMA stores clip there, the register paths mask), and the
outputs themselves checked against the oracle.
"""
import dataclasses

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
