"""Tensor-level entry points over the C ABI.

``scan_fwd`` and ``state_update`` check shapes, allocate outputs (and the
scan workspace) with torch on the inputs' device, and call the library.  They
add no arithmetic of their own.
"""
from __future__ import annotations

import torch

from . import binding as _b


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor on {device}")


def scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, initial_state=None,
             delta_softplus=True, out=None, last_state=None, workspace=None, stream=None):
    """Selective scan forward.  x, delta, z: (batch, seqlen, dim); B, C:
    (batch, seqlen, dstate); A: (dim, dstate) fp32; D, delta_bias: (dim,) fp32;
    initial_state: (batch, dim, dstate) fp32 or None.
    Returns ``(out, last_state)``."""
    if not x.is_cuda:
        raise ValueError("scan_fwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    dstate = A.shape[1]
    dev, io = x.device, x.dtype
    _check(delta, "delta", x.shape, io, dev)
    _check(z, "z", x.shape, io, dev)
    _check(B, "B", (bsz, seqlen, dstate), io, dev)
    _check(C, "C", (bsz, seqlen, dstate), io, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _check(initial_state, "initial_state", (bsz, dim, dstate), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    if last_state is None:
        last_state = torch.empty((bsz, dim, dstate), dtype=torch.float32, device=dev)
    desc = _b.make_desc(bsz, seqlen, dim, dstate, io, delta_softplus)
    need = _b.ssm_scan_workspace_size(desc)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _b.ssm_scan_fwd(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                         initial_state, workspace if need else None, wbytes if need else 0, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_scan_fwd")
    return out, last_state


def state_update(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 out=None, stream=None):
    """One decode step in place on ``state`` (batch, dim, dstate) fp32.
    x, delta, z: (batch, dim); B, C: (batch, dstate).  Returns ``out``."""
    if not state.is_cuda:
        raise ValueError("state_update runs on a CUDA device only")
    bsz, dim, dstate = state.shape
    dev, io = x.device, x.dtype
    _check(state, "state", (bsz, dim, dstate), torch.float32, dev)
    _check(x, "x", (bsz, dim), io, dev)
    _check(delta, "delta", (bsz, dim), io, dev)
    _check(z, "z", (bsz, dim), io, dev)
    _check(B, "B", (bsz, dstate), io, dev)
    _check(C, "C", (bsz, dstate), io, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    desc = _b.make_desc(bsz, 1, dim, dstate, io, delta_softplus)
    st = _b.ssm_state_update(desc, state, x, delta, A, B, C, D, z, delta_bias, out, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_state_update")
    return out
