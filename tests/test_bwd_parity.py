"""GPU parity of ssm_scan_bwd (the gradients of the scan) against the fp64
oracle's reverse-mode loop, through the C ABI.

Bounds (the pages fix none for gradients; derived from the arithmetic):
  per-token gradients dx, ddelta, dz (one value per (b, t, d), written in the
  I/O dtype): elementwise |g - g_ref| <= tol (1 + |g_ref|), tol = 1e-4 for
  fp32 I/O and 1e-2 for bf16 I/O -- the forward's bound, since each is a
  short fp32 chain like an output, rounded once to the I/O type;
  summed gradients dA, dB, dC, dD, ddelta_bias, dinitial_state (fp32 sums over
  channels, sequences or time): max |g - g_ref| <= SUM_TOL (1 + max |g_ref|)
  over the tensor -- sums of up to ~1e5 terms of mixed sign, whose error
  scales with the tensor's magnitude, not each element's.  SUM_TOL = 1e-4 for
  fp32 I/O; 1e-3 for bf16 I/O, whose path evaluates softplus and sigmoid with
  the SFU forms (relative error of Delta up to ~1e-3 where Delta ~ 1e-4, well
  inside the per-token bf16 bound), which long cancelling sums carry through.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu

SUM_TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-3}
PER_TOKEN = ("dx", "ddelta", "dz")
SUMMED = ("dA", "dB", "dC", "dD", "ddelta_bias", "dinitial_state")


def norm_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / (1.0 + np.max(np.abs(ref))))


def make_case(w, dlast=True, seed_off=500):
    inp = synth.make_scan_inputs(w)
    g = torch.Generator().manual_seed(w.seed + seed_off)
    dout = torch.randn(inp["x"].shape, generator=g).to(inp["x"].dtype)
    dl = torch.randn((w.batch, w.dim, w.dstate), generator=g) if dlast else None
    return inp, dout, dl


def check_bwd(w, cuda, dlast=True, delta_softplus=True, modify=None):
    inp, dout, dl = make_case(w, dlast)
    if modify:
        modify(inp)
    dev = to_device(inp, cuda)
    got = ops.scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dout.to(cuda),
                       D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"],
                       initial_state=dev["initial_state"],
                       dlast_state=None if dl is None else dl.to(cuda),
                       delta_softplus=delta_softplus)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                          f64(inp["C"]), f64(dout), D=f64(inp["D"]), z=f64(inp["z"]),
                          delta_bias=f64(inp["delta_bias"]), delta_softplus=delta_softplus,
                          initial_state=f64(inp["initial_state"]), dlast_state=f64(dl))
    tol = TOL[inp["x"].dtype]
    errs = {}
    for k in PER_TOKEN:
        if ref[k] is None:
            assert got[k] is None
            continue
        errs[k] = rel_err(f64(got[k]), ref[k])
        assert np.isfinite(f64(got[k])).all(), k
        assert errs[k] <= tol, f"{w.name}: {k} error {errs[k]:.3e} > {tol}"
    for k in SUMMED:
        errs[k] = norm_err(f64(got[k]), ref[k])
        assert np.isfinite(f64(got[k])).all(), k
        stol = SUM_TOL[inp["x"].dtype]
        assert errs[k] <= stol, f"{w.name}: {k} error {errs[k]:.3e} > {stol}"
    return errs


SMALL = synth.ScanWorkload("bwd-small", 2, 300, 72, 16, "bf16", 11, init_state=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_small(cuda, io):
    check_bwd(dataclasses.replace(SMALL, io=io, name=f"bwd-small-{io}"), cuda)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 32, 64])
def test_bwd_dstates(cuda, n):
    check_bwd(dataclasses.replace(SMALL, io="f32", dstate=n, seed=200 + n, name=f"bwd-n{n}"), cuda)


@pytest.mark.parametrize("variant", ["no_z", "no_D", "no_bias", "no_init", "no_dlast",
                                     "nothing_optional", "random_A", "ragged_dim"])
def test_bwd_variants(cuda, variant):
    kw = {"no_z": dict(with_z=False), "no_D": dict(with_D=False), "no_bias": dict(with_bias=False),
          "no_init": dict(init_state=False), "no_dlast": {},
          "nothing_optional": dict(with_z=False, with_D=False, with_bias=False, init_state=False),
          "random_A": dict(random_A=True), "ragged_dim": dict(dim=40, seqlen=257)}[variant]
    check_bwd(dataclasses.replace(SMALL, name=variant, seed=7, **kw), cuda,
              dlast=variant not in ("no_dlast", "nothing_optional"))


def test_bwd_without_softplus(cuda):
    def positive_delta(inp):
        inp["delta"] = (inp["delta"].float().abs() * 0.05 + 0.01).to(inp["delta"].dtype)
    check_bwd(dataclasses.replace(SMALL, name="bwd-nosoftplus", with_bias=False, seqlen=64), cuda,
              delta_softplus=False, modify=positive_delta)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 33])
def test_bwd_edge_lengths(cuda, L):
    check_bwd(dataclasses.replace(SMALL, seqlen=L, seed=40 + L, name=f"bwd-L{L}"), cuda)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_chunked_long_sequence(cuda, io):
    """Few channels and a long sequence: the time axis is cut into chunks,
    joined forward (state carries) and backward (gradient carries)."""
    w = synth.ScanWorkload(f"bwd-chunked-{io}", 1, 6000, 48, 16, io, 21, dt_lo=1e-4, dt_hi=1e-2,
                           init_state=True)
    check_bwd(w, cuda)


@pytest.mark.parametrize("n,dim", [(1, 40), (2, 40), (4, 40), (8, 40), (32, 40), (64, 40),
                                   (16, 36)])
def test_bwd_chunked_dstates(cuda, n, dim):
    """The chunked path (aggregate passes and carries) for every dstate; dim 36
    in bf16 gives rows that are not 16-byte multiples (register sweep and the
    general kernel's forward aggregate)."""
    w = synth.ScanWorkload(f"bwd-chunked-n{n}-d{dim}", 1, 3000, dim, n, "bf16" if dim == 36 else "f32",
                           300 + n, dt_lo=1e-3, dt_hi=2e-2, init_state=True)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, synth.io_dtype(w.io))
    assert binding.ssm_scan_bwd_plan(d).nchunk > 1
    check_bwd(w, cuda)


def test_bwd_empty_sequence(cuda):
    w = dataclasses.replace(SMALL, seqlen=0)
    inp, dout, dl = make_case(w)
    dev = to_device(inp, cuda)
    got = ops.scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dout.to(cuda),
                       D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"],
                       initial_state=dev["initial_state"], dlast_state=dl.to(cuda))
    torch.cuda.synchronize()
    assert torch.equal(got["dinitial_state"].cpu(), dl)
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(got[k]) == 0


def test_bwd_is_deterministic(cuda):
    w = dataclasses.replace(SMALL, seqlen=1000, dim=256, name="bwd-det")
    inp, dout, dl = make_case(w)
    dev = to_device(inp, cuda)
    args = (dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dout.to(cuda))
    kw = dict(D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"],
              initial_state=dev["initial_state"], dlast_state=dl.to(cuda))
    a = ops.scan_bwd(*args, **kw)
    b = ops.scan_bwd(*args, **kw)
    torch.cuda.synchronize()
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_bwd_full_channel_sums_medium(cuda):
    """All gradients, dB and dC included (sums over 512 channels), at a size
    the oracle finishes in seconds."""
    check_bwd(synth.ScanWorkload("bwd-medium", 2, 1024, 512, 16, "bf16", 13, init_state=True), cuda)


@pytest.mark.parametrize("mode", ["recompute", "checkpoints"])
def test_bwd_full_size_sampled_channels(cuda, mode):
    """The Mamba-1.4B layer (4 x 8192 x 4096 x 16, bf16), as the bench times it
    (7 warps of 16 channels per CTA; with the states recomputed, or read from
    the training forward's checkpoints): the per-channel gradients (dx, ddelta,
    dz over all tokens; dA, dD, ddelta_bias) of sampled channels against the
    oracle run on those channels alone (a channel's own gradients depend only
    on its own inputs and the shared B, C rows).  Channel 4095 lies in the
    partial last block (64 of 112 channels)."""
    w = synth.MAMBA_1P4B
    inp = synth.make_scan_inputs(w, device=str(cuda))
    g = torch.Generator(device=cuda).manual_seed(99)
    dout = torch.randn(inp["x"].shape, generator=g, device=cuda).to(inp["x"].dtype)
    ck = None
    if mode == "checkpoints":
        ck = ops.checkpoint_buffer(inp["x"], inp["A"])
        ops.scan_fwd(**inp, checkpoints=ck)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    assert binding.ssm_scan_bwd_plan(d, ck is not None).warps == 7
    got = ops.scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, D=inp["D"],
                       z=inp["z"], delta_bias=inp["delta_bias"], checkpoints=ck)
    torch.cuda.synchronize()
    ds = [0, 1, 2047, 4095]
    idx = torch.tensor(ds, device=cuda)
    sub = lambda t: f64(t.index_select(-1, idx))
    ref = oracle.scan_bwd(sub(inp["x"]), sub(inp["delta"]), f64(inp["A"].index_select(0, idx)),
                          f64(inp["B"]), f64(inp["C"]), sub(dout),
                          D=f64(inp["D"].index_select(0, idx)), z=sub(inp["z"]),
                          delta_bias=f64(inp["delta_bias"].index_select(0, idx)))
    tol = TOL[torch.bfloat16]
    for k in PER_TOKEN:
        e = rel_err(sub(got[k]), ref[k])
        assert e <= tol, (k, e)
    stol = SUM_TOL[torch.bfloat16]
    assert norm_err(f64(got["dA"].index_select(0, idx)), ref["dA"]) <= stol
    assert norm_err(f64(got["dD"].index_select(0, idx)), ref["dD"]) <= stol
    assert norm_err(f64(got["ddelta_bias"].index_select(0, idx)), ref["ddelta_bias"]) <= stol
    for k in ("dB", "dC"):
        assert torch.isfinite(got[k]).all()


def test_bwd_workspace_checks(cuda):
    w = SMALL
    inp, dout, dl = make_case(w)
    dev = to_device(inp, cuda)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, dev["x"].dtype)
    need = binding.ssm_scan_bwd_workspace_size(desc)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=cuda)
    outs = [torch.empty_like(dev["x"]) for _ in range(2)]
    f = lambda *s: torch.empty(s, device=cuda)
    st = binding.ssm_scan_bwd(desc, dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], None,
                              None, None, None, dout.to(cuda), None, outs[0], outs[1],
                              f(w.dim, w.dstate), f(w.batch, w.seqlen, w.dstate),
                              f(w.batch, w.seqlen, w.dstate), None, None, None, None, small,
                              small.numel())
    assert st == binding.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("case", ["small-bf16", "small-f32", "chunked", "n8", "ragged"])
def test_bwd_with_training_checkpoints(cuda, case):
    """The training pair: the forward keeps the state before every 16th
    token; the checkpoints match the oracle's states there; the backward that
    reads them matches the oracle's gradients."""
    w = {"small-bf16": SMALL, "small-f32": dataclasses.replace(SMALL, io="f32"),
         "chunked": synth.ScanWorkload("ck-chunked", 1, 6000, 48, 16, "bf16", 21, dt_lo=1e-4,
                                       dt_hi=1e-2, init_state=True),
         "n8": dataclasses.replace(SMALL, dstate=8, io="f32", seed=5),
         "ragged": dataclasses.replace(SMALL, dim=40, seqlen=257, seed=6)}[case]
    inp, dout, dl = make_case(w)
    dev = to_device(inp, cuda)
    ck = ops.checkpoint_buffer(dev["x"], dev["A"])
    ops.scan_fwd(**dev, checkpoints=ck)
    torch.cuda.synchronize()
    ntiles = (w.seqlen + 15) // 16
    ckv = ck[: w.batch * ntiles * w.dim * w.dstate].view(w.batch, ntiles, w.dim, w.dstate)
    tol = TOL[inp["x"].dtype]
    for j in sorted({0, 1, ntiles // 2, ntiles - 1}):
        cut = lambda t: None if t is None else t[:, :16 * j]
        if j == 0:
            ref_state = f64(inp["initial_state"])
        else:
            _, ref_state = oracle.scan_fwd(f64(cut(inp["x"])), f64(cut(inp["delta"])), f64(inp["A"]),
                                           f64(cut(inp["B"])), f64(cut(inp["C"])), D=f64(inp["D"]),
                                           z=f64(cut(inp["z"])), delta_bias=f64(inp["delta_bias"]),
                                           initial_state=f64(inp["initial_state"]))
        assert rel_err(f64(ckv[:, j]), ref_state) <= tol, j
    got = ops.scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dout.to(cuda),
                       D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"],
                       initial_state=dev["initial_state"], dlast_state=dl.to(cuda), checkpoints=ck)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                          f64(inp["C"]), f64(dout), D=f64(inp["D"]), z=f64(inp["z"]),
                          delta_bias=f64(inp["delta_bias"]), initial_state=f64(inp["initial_state"]),
                          dlast_state=f64(dl))
    for k in PER_TOKEN:
        assert rel_err(f64(got[k]), ref[k]) <= tol, k
    for k in SUMMED:
        assert norm_err(f64(got[k]), ref[k]) <= SUM_TOL[inp["x"].dtype], k


def test_bwd_unaligned_tensors(cuda):
    """Token tensors whose base addresses are not 16-byte aligned (a storage
    offset of one element): the dstate-16 backward falls back from the TMA
    sweeps to the register sweep, in the same workspace, with the same
    gradients."""
    w = dataclasses.replace(SMALL, name="bwd-unaligned", seed=17)
    inp, dout, dl = make_case(w)
    dev = to_device(inp, cuda)

    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=cuda)
        v = buf[1:1 + t.numel()].view(t.shape)
        v.copy_(t.to(cuda))
        assert v.data_ptr() % 16 != 0
        return v
    for k in ("x", "delta", "z"):
        dev[k] = shifted(dev[k])
    got = ops.scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], shifted(dout),
                       D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"],
                       initial_state=dev["initial_state"], dlast_state=dl.to(cuda))
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(inp["x"]), f64(inp["delta"]), f64(inp["A"]), f64(inp["B"]),
                          f64(inp["C"]), f64(dout), D=f64(inp["D"]), z=f64(inp["z"]),
                          delta_bias=f64(inp["delta_bias"]), initial_state=f64(inp["initial_state"]),
                          dlast_state=f64(dl))
    for k in PER_TOKEN:
        assert rel_err(f64(got[k]), ref[k]) <= TOL[torch.bfloat16], k
    for k in SUMMED:
        assert norm_err(f64(got[k]), ref[k]) <= SUM_TOL[torch.bfloat16], k


def shape_for_warps(warps, n, io, L=40):
    """The smallest (batch, dim) whose backward plan sweeps in one chunk with
    `warps` warps per CTA and, where the channel block allows it, a partial
    last block of channels (found through the plan query)."""
    dt = synth.io_dtype(io)
    for total in range(8, 60000, 8):
        for b in (1, 2, 4):
            if total % b or (total // b) % 8:
                continue
            d = total // b
            pl = binding.ssm_scan_bwd_plan(binding.make_desc(b, L, d, n, dt))
            if pl.nchunk == 1 and pl.warps == warps and (d % pl.channels or pl.channels <= 8):
                return b, d
    raise AssertionError(f"no shape selects {warps} warps at dstate {n}")


@pytest.mark.parametrize("n,warps,io", [(16, 1, "bf16"), (16, 2, "bf16"), (16, 3, "f32"),
                                        (16, 4, "bf16"), (16, 5, "bf16"), (16, 6, "bf16"),
                                        (16, 6, "f32"), (16, 7, "bf16"), (8, 5, "bf16"),
                                        (8, 7, "f32"), (32, 6, "bf16"), (64, 4, "bf16")])
def test_bwd_warps_per_cta(cuda, n, warps, io):
    """Every CTA width of the reverse sweeps, on a shape that selects it (one
    chunk; 40 steps = two full tiles and a ragged one; a partial last block of
    channels where the width allows one).  dstate 16 runs the one-warp-layout
    sweep (CTAs of 1..7 warps, 16 channels each; the width of a single warp
    with 8 channels is the smallest case), the other dstates the sweep of
    8 channels a warp."""
    b, d = shape_for_warps(warps, n, io)
    w = synth.ScanWorkload(f"bwd-w{warps}-n{n}-{io}", b, 40, d, n, io, 30 + warps + n,
                           init_state=True)
    check_bwd(w, cuda)
