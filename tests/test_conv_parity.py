"""GPU parity of the causal depthwise conv (+ SiLU) entry points against the
fp64 oracle, through the C ABI:

  ssm_conv1d_fwd        vs oracle.conv1d_fwd
  ssm_conv_scan_fwd     vs oracle.conv1d_fwd followed by oracle.scan_fwd on x_conv
  ssm_conv_state_update vs the same two oracle calls, one token at a time

Bounds: |y - y_ref| <= tol (1 + |y_ref|), tol = 1e-4 for fp32 I/O and 1e-2 for
bf16 I/O, for outputs and SSM states.  The conv state that comes out is a
copy of raw inputs (or of the incoming state), so it must match exactly."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu


def oracle_conv_scan(inp, conv, activation=True, delta_softplus=True):
    """x_conv from the oracle conv, then the oracle scan on it."""
    xc, cst = oracle.conv1d_fwd(f64(inp["x"]), f64(conv["conv_w"]), f64(conv["conv_bias"]),
                                f64(conv["conv_state"]), activation)
    out, last = oracle.scan_fwd(xc, f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]), f64(inp["C"]),
                                D=f64(inp["D"]), z=f64(inp["z"]), delta_bias=f64(inp["delta_bias"]),
                                delta_softplus=delta_softplus,
                                initial_state=f64(inp["initial_state"]))
    return out, last, cst


# ---------------------------------------------------------------- conv alone

@pytest.mark.parametrize("width", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dim", [72, 36])          # 36: rows not a 16-byte multiple in bf16
def test_conv1d_widths(cuda, width, io, dim):
    bsz, L = 2, 300
    w = synth.ScanWorkload("conv", bsz, L, dim, 1, io, 60 + width)
    x = synth.make_scan_inputs(w)["x"]
    conv = synth.make_conv_inputs(bsz, dim, width, seed=70 + width, with_state=True)
    xd, cd = x.to(cuda), to_device(conv, cuda)
    out, st = ops.conv1d_fwd(xd, cd["conv_w"], cd["conv_bias"], cd["conv_state"])
    torch.cuda.synchronize()
    ref, ref_st = oracle.conv1d_fwd(f64(x), f64(conv["conv_w"]), f64(conv["conv_bias"]),
                                    f64(conv["conv_state"]), True)
    assert rel_err(f64(out), ref) <= TOL[x.dtype]
    assert np.array_equal(f64(st), ref_st)


@pytest.mark.parametrize("variant", ["no_bias", "no_state", "no_act", "short", "one_step"])
def test_conv1d_variants(cuda, variant):
    bsz, dim, width = 3, 64, 4
    L = {"short": 2, "one_step": 1}.get(variant, 129)       # short: fewer steps than K-1
    w = synth.ScanWorkload("conv", bsz, L, dim, 1, "bf16", 80)
    x = synth.make_scan_inputs(w)["x"]
    conv = synth.make_conv_inputs(bsz, dim, width, seed=81, with_bias=variant != "no_bias",
                                  with_state=variant != "no_state")
    act = variant != "no_act"
    xd, cd = x.to(cuda), to_device(conv, cuda)
    out, st = ops.conv1d_fwd(xd, cd["conv_w"], cd["conv_bias"], cd["conv_state"], activation=act)
    torch.cuda.synchronize()
    ref, ref_st = oracle.conv1d_fwd(f64(x), f64(conv["conv_w"]), f64(conv["conv_bias"]),
                                    f64(conv["conv_state"]), act)
    assert rel_err(f64(out), ref) <= TOL[x.dtype]
    assert np.array_equal(f64(st), ref_st)


def test_conv1d_empty_sequence_copies_state(cuda):
    conv = to_device(synth.make_conv_inputs(2, 32, 4, seed=3, with_state=True), cuda)
    x = torch.empty(2, 0, 32, device=cuda, dtype=torch.bfloat16)
    out, st = ops.conv1d_fwd(x, conv["conv_w"], conv["conv_bias"], conv["conv_state"])
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(st, conv["conv_state"])


def test_conv1d_chunks_agree_with_one_pass(cuda):
    """Feeding the sequence in two pieces, the conv state carried between
    them, gives the one-pass result exactly (same fp32 arithmetic per token)."""
    bsz, L, dim, width = 2, 1000, 128, 4
    x = synth.make_scan_inputs(synth.ScanWorkload("c", bsz, L, dim, 1, "f32", 90))["x"].to(cuda)
    conv = to_device(synth.make_conv_inputs(bsz, dim, width, seed=91, with_state=True), cuda)
    full, st = ops.conv1d_fwd(x, conv["conv_w"], conv["conv_bias"], conv["conv_state"])
    a, st_a = ops.conv1d_fwd(x[:, :377].contiguous(), conv["conv_w"], conv["conv_bias"],
                             conv["conv_state"])
    b, st_b = ops.conv1d_fwd(x[:, 377:].contiguous(), conv["conv_w"], conv["conv_bias"], st_a)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([a, b], 1), full) and torch.equal(st_b, st)


# ------------------------------------------------------------- conv + scan

SMALL = synth.ScanWorkload("conv-scan-bf16", 2, 300, 72, 16, "bf16", 11, init_state=True)


def check_conv_scan(w, cuda, width=4, activation=True, with_state=True, with_bias=True):
    inp = synth.make_scan_inputs(w)
    conv = synth.make_conv_inputs(w.batch, w.dim, width, seed=w.seed + 1000,
                                  with_bias=with_bias, with_state=with_state)
    dev, cd = to_device(inp, cuda), to_device(conv, cuda)
    out, last, cst = ops.conv_scan_fwd(dev["x"], cd["conv_w"], dev["delta"], dev["A"], dev["B"],
                                       dev["C"], D=dev["D"], z=dev["z"],
                                       delta_bias=dev["delta_bias"], conv_bias=cd["conv_bias"],
                                       conv_state=cd["conv_state"],
                                       initial_state=dev["initial_state"], activation=activation)
    torch.cuda.synchronize()
    ref, ref_last, ref_cst = oracle_conv_scan(inp, conv, activation)
    tol = TOL[inp["x"].dtype]
    e_out, e_last = rel_err(f64(out), ref), rel_err(f64(last), ref_last)
    assert np.isfinite(f64(out)).all()
    assert e_out <= tol, f"{w.name} K={width}: out error {e_out:.3e} > {tol}"
    assert e_last <= tol, f"{w.name} K={width}: last_state error {e_last:.3e} > {tol}"
    assert np.array_equal(f64(cst), ref_cst), f"{w.name} K={width}: conv state differs"
    return e_out, e_last


@pytest.mark.parametrize("width", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_scan_widths(cuda, width, io):
    check_conv_scan(dataclasses.replace(SMALL, io=io, seed=20 + width), cuda, width=width)


@pytest.mark.parametrize("n", [4, 8, 16, 32])
def test_conv_scan_dstates(cuda, n):
    """dstate 16 takes the warp-specialised kernel, the others the generic one."""
    check_conv_scan(dataclasses.replace(SMALL, dstate=n, seed=30 + n), cuda)


@pytest.mark.parametrize("variant", ["no_act", "no_state", "no_bias", "ragged_dim",
                                     "narrow_rows", "nothing_optional"])
def test_conv_scan_variants(cuda, variant):
    kw, ckw = {}, {}
    if variant == "no_act":
        ckw = dict(activation=False)
    elif variant == "no_state":
        ckw = dict(with_state=False)
    elif variant == "no_bias":
        ckw = dict(with_bias=False)
    elif variant == "ragged_dim":
        kw = dict(dim=40, seqlen=257)             # last CTA half full, ragged time tail
    elif variant == "narrow_rows":
        kw = dict(dim=12)                         # 24-byte bf16 rows: generic kernel
    elif variant == "nothing_optional":
        kw = dict(with_z=False, with_D=False, with_bias=False, init_state=False)
        ckw = dict(with_state=False, with_bias=False)
    check_conv_scan(dataclasses.replace(SMALL, name=variant, seed=7, **kw), cuda, **ckw)


@pytest.mark.parametrize("L", [1, 2, 3, 17, 33])
def test_conv_scan_edge_lengths(cuda, L):
    """Sequences shorter than the conv history (the state supplies the rest)
    and ragged tile tails."""
    check_conv_scan(dataclasses.replace(SMALL, seqlen=L, seed=40 + L), cuda, width=4)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_scan_chunked_long_sequence(cuda, io):
    """Long sequence, few channels: the time axis is cut into chunks; every
    chunk's conv reaches back into the previous chunk's raw inputs."""
    w = synth.ScanWorkload(f"conv-chunked-{io}", 1, 6000, 48, 16, io, 21, dt_lo=1e-4,
                           dt_hi=1e-2, init_state=True)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, synth.io_dtype(io))
    assert binding.ssm_scan_plan(d).nchunk > 1, "case meant to exercise the chunked path"
    check_conv_scan(w, cuda, width=4)


def test_conv_scan_generic_chunked(cuda):
    """The generic kernel's chunked mode with the conv (dstate 4)."""
    w = synth.ScanWorkload("conv-chunked-n4", 1, 6000, 24, 4, "f32", 22, dt_lo=1e-4,
                           dt_hi=1e-2, init_state=True)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, torch.float32)
    assert binding.ssm_scan_plan(d).path == 0 and binding.ssm_scan_plan(d).nchunk > 1
    check_conv_scan(w, cuda, width=3)


def test_conv_scan_empty_sequence(cuda):
    w = dataclasses.replace(SMALL, seqlen=0)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    conv = to_device(synth.make_conv_inputs(w.batch, w.dim, 4, seed=5, with_state=True), cuda)
    out, last, cst = ops.conv_scan_fwd(inp["x"], conv["conv_w"], inp["delta"], inp["A"], inp["B"],
                                       inp["C"], D=inp["D"], z=inp["z"],
                                       delta_bias=inp["delta_bias"], conv_state=conv["conv_state"],
                                       initial_state=inp["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(last, inp["initial_state"]) and torch.equal(cst, conv["conv_state"])


def test_conv_scan_matches_conv_then_scan_on_gpu(cuda):
    """Fused == the two separate library calls with fp32 I/O (x_conv is
    then stored exactly, so only rounding order differs)."""
    w = dataclasses.replace(SMALL, io="f32", seed=99)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    conv = to_device(synth.make_conv_inputs(w.batch, w.dim, 4, seed=98, with_state=True), cuda)
    xc, cst_sep = ops.conv1d_fwd(inp["x"], conv["conv_w"], conv["conv_bias"], conv["conv_state"])
    sep, sep_last = ops.scan_fwd(**dict(inp, x=xc))
    fused, f_last, cst = ops.conv_scan_fwd(inp["x"], conv["conv_w"], inp["delta"], inp["A"],
                                           inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                                           delta_bias=inp["delta_bias"],
                                           conv_bias=conv["conv_bias"],
                                           conv_state=conv["conv_state"],
                                           initial_state=inp["initial_state"])
    torch.cuda.synchronize()
    assert rel_err(f64(fused), f64(sep)) <= 1e-5
    assert rel_err(f64(f_last), f64(sep_last)) <= 1e-5
    assert torch.equal(cst, cst_sep)


# ------------------------------------------------------------- decode + conv

def element_aligned(t):
    """t's values one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


def run_conv_decode_chain(cuda, n, io, width, shift=False):
    bsz, dim, steps = 3, 72, 8
    w = synth.DecodeWorkload("conv-decode", bsz, dim, n, steps, io, 140 + n + 7 * width)
    inp = synth.make_decode_inputs(w)
    conv = synth.make_conv_inputs(bsz, dim, width, seed=150 + n + width, with_state=True)
    dev, cd = to_device(inp, cuda), to_device(conv, cuda)
    if shift:   # element loads instead of vector loads for A, B, C
        dev = dict(dev, A=element_aligned(dev["A"]), B=element_aligned(dev["B"]),
                   C=element_aligned(dev["C"]))
    tol = TOL[synth.io_dtype(io)]
    state, cstate = dev["state"].clone(), cd["conv_state"].clone()
    ref_state, ref_cstate = f64(inp["state"]), f64(conv["conv_state"])
    for s in range(steps):
        out = ops.conv_state_update(cstate, cd["conv_w"], state, dev["x"][s], dev["delta"][s],
                                    dev["A"], dev["B"][s], dev["C"][s], D=dev["D"], z=dev["z"][s],
                                    delta_bias=dev["delta_bias"], conv_bias=cd["conv_bias"])
        torch.cuda.synchronize()
        xc, ref_cstate = oracle.conv1d_fwd(f64(inp["x"][s])[:, None, :], f64(conv["conv_w"]),
                                           f64(conv["conv_bias"]), ref_cstate, True)
        ref_out, ref_state = oracle.state_update(ref_state, xc[:, 0, :], f64(inp["delta"][s]),
                                                 f64(inp["A"]), f64(inp["B"][s]), f64(inp["C"][s]),
                                                 f64(inp["D"]), f64(inp["z"][s]),
                                                 f64(inp["delta_bias"]))
        assert rel_err(f64(out), ref_out) <= tol, (s, rel_err(f64(out), ref_out))
        assert rel_err(f64(state), ref_state) <= tol
        assert np.array_equal(f64(cstate), ref_cstate), s


@pytest.mark.parametrize("n", [1, 4, 16, 64])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_decode_chain(cuda, n, io):
    """Width 4 (the kernel with the width fixed at compile time)."""
    run_conv_decode_chain(cuda, n, io, 4)


@pytest.mark.parametrize("width", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("n", [4, 16])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_decode_widths(cuda, width, n, io):
    """Other widths take the runtime-width kernel: histories that fit the
    channel's lanes (shuffle shift) and longer ones (per-lane reads)."""
    run_conv_decode_chain(cuda, n, io, width)


@pytest.mark.parametrize("width", [3, 4])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_decode_element_aligned(cuda, width, io):
    run_conv_decode_chain(cuda, 16, io, width, shift=True)


def test_conv_decode_continues_prefill(cuda):
    """Prefill with the fused conv+scan over L tokens, then decode token L+1
    with the returned conv and SSM states == the fused prefill over L+1."""
    w = dataclasses.replace(SMALL, seqlen=65, seed=12)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    conv = to_device(synth.make_conv_inputs(w.batch, w.dim, 4, seed=13, with_state=True), cuda)
    kw = dict(conv_bias=conv["conv_bias"], conv_state=conv["conv_state"],
              initial_state=inp["initial_state"])
    full, full_last, full_cst = ops.conv_scan_fwd(inp["x"], conv["conv_w"], inp["delta"], inp["A"],
                                                  inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                                                  delta_bias=inp["delta_bias"], **kw)
    cut = lambda t: t[:, :64].contiguous()
    _, last, cst = ops.conv_scan_fwd(cut(inp["x"]), conv["conv_w"], cut(inp["delta"]), inp["A"],
                                     cut(inp["B"]), cut(inp["C"]), D=inp["D"], z=cut(inp["z"]),
                                     delta_bias=inp["delta_bias"], **kw)
    y = ops.conv_state_update(cst, conv["conv_w"], last, inp["x"][:, 64].contiguous(),
                              inp["delta"][:, 64].contiguous(), inp["A"],
                              inp["B"][:, 64].contiguous(), inp["C"][:, 64].contiguous(),
                              D=inp["D"], z=inp["z"][:, 64].contiguous(),
                              delta_bias=inp["delta_bias"], conv_bias=conv["conv_bias"])
    torch.cuda.synchronize()
    tol = TOL[torch.bfloat16]
    assert rel_err(f64(y), f64(full[:, 64])) <= tol
    assert rel_err(f64(last), f64(full_last)) <= tol
    assert torch.equal(cst, full_cst)


# ------------------------------------------------------------ full size, sampled

def test_conv_full_size_sampled(cuda):
    """The Mamba-1.4B layer (4 x 8192 x 4096, bf16) with the width-4 conv and
    the inputs the benchmark draws: the standalone conv (TMA-streamed) and the
    fused conv + scan, on sampled channels of sampled sequences (all 8192
    tokens), against the oracle conv and scan run on those channels alone."""
    from parity import sample_channels
    w = synth.MAMBA_1P4B
    inp = synth.make_scan_inputs(w, device=str(cuda))
    conv = synth.make_conv_inputs(w.batch, w.dim, 4, seed=w.seed + 500, device=str(cuda))
    xc, cst = ops.conv1d_fwd(inp["x"], conv["conv_w"], conv["conv_bias"], None)
    out, last, cst2 = ops.conv_scan_fwd(inp["x"], conv["conv_w"], inp["delta"], inp["A"], inp["B"],
                                        inp["C"], D=inp["D"], z=inp["z"],
                                        delta_bias=inp["delta_bias"], conv_bias=conv["conv_bias"])
    torch.cuda.synchronize()
    tol = TOL[inp["x"].dtype]
    for b, ds in sample_channels(w.batch, w.dim):
        idx = torch.tensor(ds, device=cuda)
        tok = lambda t: f64(t[b].index_select(-1, idx))[None]       # (1, L, nd)
        par = lambda t: f64(t.index_select(0, idx))
        ref_xc, ref_cst = oracle.conv1d_fwd(tok(inp["x"]), par(conv["conv_w"]),
                                            par(conv["conv_bias"]), None, True)
        assert rel_err(tok(xc), ref_xc) <= tol, (b, ds)
        assert np.array_equal(f64(cst[b].index_select(0, idx))[None], ref_cst), (b, ds)
        ref_out, ref_last = oracle.scan_fwd(ref_xc, tok(inp["delta"]), par(inp["A"]),
                                            f64(inp["B"][b])[None], f64(inp["C"][b])[None],
                                            D=par(inp["D"]), z=tok(inp["z"]),
                                            delta_bias=par(inp["delta_bias"]))
        assert rel_err(tok(out), ref_out) <= tol, (b, ds, rel_err(tok(out), ref_out))
        assert rel_err(f64(last[b].index_select(0, idx))[None], ref_last) <= tol, (b, ds)
        assert np.array_equal(f64(cst2[b].index_select(0, idx))[None], ref_cst), (b, ds)


def test_conv_decode_full_size_sampled(cuda):
    """The decode shape (256 sequences x 5120 channels, dstate 16, bf16) with
    the width-4 conv in front, as the benchmark times it (the compile-time
    width kernel): 4 chained steps, sampled channels against the oracle's conv
    step and decode step run on those channels alone."""
    from parity import sample_channels
    w = synth.DECODE
    inp = synth.make_decode_inputs(w, device=str(cuda))
    conv = synth.make_conv_inputs(w.batch, w.dim, 4, seed=w.seed + 3, device=str(cuda),
                                  with_state=True)
    state, cstate = inp["state"].clone(), conv["conv_state"].clone()
    samples = sample_channels(w.batch, w.dim)
    refs = {}
    for b, ds in samples:
        idx = torch.tensor(ds, device=cuda)
        refs[b] = (f64(inp["state"][b].index_select(0, idx))[None],
                   f64(conv["conv_state"][b].index_select(0, idx))[None])
    tol = TOL[inp["x"].dtype]
    for s in range(4):
        out = ops.conv_state_update(cstate, conv["conv_w"], state, inp["x"][s], inp["delta"][s],
                                    inp["A"], inp["B"][s], inp["C"][s], D=inp["D"], z=inp["z"][s],
                                    delta_bias=inp["delta_bias"], conv_bias=conv["conv_bias"])
        torch.cuda.synchronize()
        for b, ds in samples:
            idx = torch.tensor(ds, device=cuda)
            par = lambda t: f64(t.index_select(0, idx))
            row = lambda t: f64(t[s][b].index_select(0, idx))[None]    # (1, nd)
            ref_h, ref_c = refs[b]
            xc, ref_c = oracle.conv1d_fwd(row(inp["x"])[:, None, :], par(conv["conv_w"]),
                                          par(conv["conv_bias"]), ref_c, True)
            ref_out, ref_h = oracle.state_update(ref_h, xc[:, 0, :], row(inp["delta"]), par(inp["A"]),
                                                 f64(inp["B"][s][b])[None], f64(inp["C"][s][b])[None],
                                                 par(inp["D"]), row(inp["z"]), par(inp["delta_bias"]))
            refs[b] = (ref_h, ref_c)
            assert rel_err(f64(out[b].index_select(0, idx))[None], ref_out) <= tol, (s, b, ds)
            assert rel_err(f64(state[b].index_select(0, idx))[None], ref_h) <= tol, (s, b, ds)
            assert np.array_equal(f64(cstate[b].index_select(0, idx))[None], ref_c), (s, b, ds)
