"""GPU parity of ssm_scan_fwd against the fp64 oracle (called through the
C ABI), elementwise, within |y - y_ref| <= tol (1 + |y_ref|): tol = 1e-4 for
fp32 I/O and 1e-2 for bf16 I/O, the same bound for the final state."""
import dataclasses

import numpy as np
import pytest
import torch

from parity import TOL, f64, oracle_full, oracle_sampled, rel_err, sample_channels, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu


def check_full(w, cuda, delta_softplus=True, modify=None):
    inp = synth.make_scan_inputs(w)
    if modify:
        modify(inp)
    dev = to_device(inp, cuda)
    out, last = ops.scan_fwd(**dev, delta_softplus=delta_softplus)
    torch.cuda.synchronize()
    ref, ref_last = oracle_full(inp, delta_softplus)
    tol = TOL[inp["x"].dtype]
    e_out, e_last = rel_err(f64(out), ref), rel_err(f64(last), ref_last)
    assert np.isfinite(f64(out)).all()
    assert e_out <= tol, f"{w.name}: out error {e_out:.3e} > {tol}"
    assert e_last <= tol, f"{w.name}: last_state error {e_last:.3e} > {tol}"
    return e_out, e_last


def test_tiny_fp32(cuda):
    check_full(synth.TINY, cuda)


SMALL = synth.ScanWorkload("small-bf16", 2, 300, 72, 16, "bf16", 11)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_dstate_and_dtype(cuda, n, io):
    w = dataclasses.replace(SMALL, dstate=n, io=io, seed=100 + n, name=f"small-{io}-n{n}")
    check_full(w, cuda)


@pytest.mark.parametrize("variant", ["random_A", "init_state", "no_z", "no_D", "no_bias",
                                     "nothing_optional", "ragged_dim"])
def test_variants(cuda, variant):
    kw = {"random_A": dict(random_A=True), "init_state": dict(init_state=True),
          "no_z": dict(with_z=False), "no_D": dict(with_D=False), "no_bias": dict(with_bias=False),
          "nothing_optional": dict(with_z=False, with_D=False, with_bias=False),
          "ragged_dim": dict(dim=40, seqlen=257)}[variant]
    check_full(dataclasses.replace(SMALL, name=variant, seed=7, **kw), cuda)


def test_without_softplus(cuda):
    def positive_delta(inp):
        inp["delta"] = (inp["delta"].float().abs() * 0.05 + 0.01).to(inp["delta"].dtype)
    check_full(dataclasses.replace(SMALL, name="nosoftplus", with_bias=False, seqlen=64), cuda,
               delta_softplus=False, modify=positive_delta)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunked_long_sequence(cuda, io):
    """Few channels and a long sequence: the time axis is cut into chunks
    joined by the carry pass; compared in full against the oracle."""
    w = synth.ScanWorkload(f"chunked-{io}", 1, 6000, 48, 16, io, 21, dt_lo=1e-4, dt_hi=1e-2,
                           init_state=True)
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, synth.io_dtype(io))
    assert binding.ssm_scan_workspace_size(d) > 0, "case meant to exercise the chunked path"
    check_full(w, cuda)


def test_edge_lengths(cuda):
    for L in (1, 2, 31, 33):
        check_full(dataclasses.replace(SMALL, seqlen=L, name=f"L{L}", init_state=True), cuda)


def test_empty_sequence_copies_state(cuda):
    w = dataclasses.replace(SMALL, seqlen=0, init_state=True)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    out, last = ops.scan_fwd(**inp)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(last, inp["initial_state"])
    inp["initial_state"] = None
    _, last = ops.scan_fwd(**inp)
    assert torch.count_nonzero(last).item() == 0


def test_split_and_carry(cuda):
    """[0, L1) then [L1, L) from the first call's last_state equals one call."""
    w = dataclasses.replace(SMALL, seqlen=400, init_state=True, seed=31)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    out, last = ops.scan_fwd(**inp)
    cut = lambda sl: {k: (v[:, sl].contiguous() if k in ("x", "delta", "z", "B", "C") else v)
                      for k, v in inp.items()}
    o1, l1 = ops.scan_fwd(**cut(slice(0, 123)))
    p2 = cut(slice(123, None))
    p2["initial_state"] = l1
    o2, l2 = ops.scan_fwd(**p2)
    torch.cuda.synchronize()
    assert rel_err(f64(torch.cat([o1, o2], 1)), f64(out)) <= TOL[torch.bfloat16]
    assert rel_err(f64(l2), f64(last)) <= TOL[torch.bfloat16]


def test_no_write_outside_outputs(cuda):
    """Outputs live inside larger buffers filled with a sentinel; nothing
    outside the described tensors may change."""
    w = dataclasses.replace(SMALL, seqlen=97, dim=40, init_state=True)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    n_out, n_st = inp["x"].numel(), inp["initial_state"].numel()
    big_out = torch.full((n_out + 4096,), -77.0, dtype=inp["x"].dtype, device=cuda)
    big_st = torch.full((n_st + 1024,), -77.0, dtype=torch.float32, device=cuda)
    out = big_out[:n_out].view_as(inp["x"])
    last = big_st[:n_st].view_as(inp["initial_state"])
    ops.scan_fwd(**inp, out=out, last_state=last)
    torch.cuda.synchronize()
    assert torch.all(big_out[n_out:] == -77.0) and torch.all(big_st[n_st:] == -77.0)
    ref, ref_last = oracle_full(synth.make_scan_inputs(w))
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]


def test_rejects_misaligned_and_leaves_output(cuda):
    w = dataclasses.replace(SMALL, seqlen=16)
    inp = to_device(synth.make_scan_inputs(w), cuda)
    out = torch.full_like(inp["x"], 5.0)
    x_off = inp["x"].data_ptr() + 1          # a bf16 tensor at an odd address
    d = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    st = binding.ssm_scan_fwd(d, x_off, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["delta_bias"], out, None, None, None, 0)
    torch.cuda.synchronize()
    assert st == binding.SSM_ERR_INVALID_ARG
    assert torch.all(out == 5.0)


@pytest.mark.parametrize("w", [synth.MAMBA_130M, synth.MAMBA_1P4B, synth.LONG_SEQ],
                         ids=lambda w: w.name)
def test_full_size_sampled(cuda, w):
    """Full-size Mamba-shaped workloads in the same launch configuration the
    benchmark times; every output of sampled channels (all L tokens) and their
    final states are compared with the oracle."""
    inp = synth.make_scan_inputs(w, device=str(cuda))
    out, last = ops.scan_fwd(**inp)
    torch.cuda.synchronize()
    tol = TOL[inp["x"].dtype]
    assert torch.isfinite(out.float()).all()
    for b, (ds, ref, ref_last) in oracle_sampled(inp, sample_channels(w.batch, w.dim)).items():
        idx = torch.tensor(ds, device=cuda)
        got = f64(out[b].index_select(-1, idx))
        got_last = f64(last[b].index_select(0, idx))
        assert rel_err(got, ref) <= tol, (b, ds, rel_err(got, ref))
        assert rel_err(got_last, ref_last) <= tol, (b, ds, rel_err(got_last, ref_last))


def _misaligned_copy(t, cuda):
    """Same values at an address that is element-aligned but not 16-byte aligned."""
    e = t.element_size()
    off = 8 // e
    buf = torch.empty(t.numel() + off, dtype=t.dtype, device=cuda)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0
    return v


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_general_path_when_not_16_byte_aligned(cuda, io):
    """Element-aligned but not 16-byte aligned tensors take the general kernel;
    it must agree with the oracle too (dstate 16, the tiled path's shape)."""
    w = dataclasses.replace(SMALL, io=io, init_state=True, seed=81)
    inp = synth.make_scan_inputs(w)
    dev = to_device(inp, cuda)
    for k in ("x", "delta", "z"):
        dev[k] = _misaligned_copy(dev[k], cuda)
    out = _misaligned_copy(torch.zeros_like(dev["x"]), cuda)
    out, last = ops.scan_fwd(**dev, out=out)
    torch.cuda.synchronize()
    ref, ref_last = oracle_full(inp)
    tol = TOL[inp["x"].dtype]
    assert rel_err(f64(out), ref) <= tol and rel_err(f64(last), ref_last) <= tol


def test_tiled_and_general_paths_agree(cuda):
    w = dataclasses.replace(SMALL, seqlen=700, init_state=True, seed=82)
    dev = to_device(synth.make_scan_inputs(w), cuda)
    out_t, last_t = ops.scan_fwd(**dev)
    mis = dict(dev)
    for k in ("x", "delta", "z"):
        mis[k] = _misaligned_copy(dev[k], cuda)
    out_g, last_g = ops.scan_fwd(**mis, out=_misaligned_copy(torch.zeros_like(dev["x"]), cuda))
    torch.cuda.synchronize()
    assert rel_err(f64(out_t), f64(out_g)) <= 1e-2
    assert rel_err(f64(last_t), f64(last_g)) <= 1e-3
