"""Tensor-level entry points over the C ABI.

``scan_fwd``, ``scan_bwd`` (its gradients), ``state_update`` and the conv
variants (``conv1d_fwd``, ``conv_scan_fwd``, ``conv_state_update``) check shapes, allocate outputs (and
the scan workspace) with torch on the inputs' device, and call the library.
They add no arithmetic of their own.
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
             delta_softplus=True, out=None, last_state=None, workspace=None, stream=None,
             discretization="euler", checkpoints=None):
    """Selective scan forward.  x, delta, z: (batch, seqlen, dim); B, C:
    (batch, seqlen, dstate); A: (dim, dstate) fp32; D, delta_bias: (dim,) fp32;
    initial_state: (batch, dim, dstate) fp32 or None.  ``discretization``:
    "euler" (input term Delta B x) or "zoh" (exact zero-order hold).
    ``checkpoints``: an fp32 device buffer of ssm_scan_checkpoint_size bytes
    to keep the state before every 16th token for scan_bwd (training).
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
    if checkpoints is not None and discretization != "euler":
        raise ValueError("checkpoints are kept by the first-order scan only")
    if discretization == "euler":
        st = _b.ssm_scan_fwd(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                             initial_state, workspace if need else None, wbytes if need else 0,
                             stream) if checkpoints is None else \
        _b.ssm_scan_fwd_train(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                              initial_state, checkpoints, workspace if need else None,
                              wbytes if need else 0, stream)
    else:
        st = _b.ssm_scan_fwd_ex(desc, _b.make_opts(discretization), x, delta, A, B, C, D, z,
                                delta_bias, out, last_state, initial_state,
                                workspace if need else None, wbytes if need else 0, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_scan_fwd")
    return out, last_state


def state_update(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 out=None, stream=None, discretization="euler"):
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
    if discretization == "euler":
        st = _b.ssm_state_update(desc, state, x, delta, A, B, C, D, z, delta_bias, out, stream)
    else:
        st = _b.ssm_state_update_ex(desc, _b.make_opts(discretization), state, x, delta, A, B, C,
                                    D, z, delta_bias, out, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_state_update")
    return out


def _conv_state_shape(bsz, dim, width):
    return (bsz, dim, width - 1)


def conv1d_fwd(x, w, bias=None, conv_state=None, activation=True, out=None,
               conv_state_out=None, stream=None):
    """Causal depthwise conv of x (batch, seqlen, dim) with taps w (dim, width)
    fp32, optional bias (dim,), optional history conv_state (batch, dim,
    width-1) fp32.  Returns ``(x_conv, conv_state_out)``."""
    if not x.is_cuda:
        raise ValueError("conv1d_fwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    width = w.shape[1]
    dev = x.device
    _check(w, "w", (dim, width), torch.float32, dev)
    _check(bias, "bias", (dim,), torch.float32, dev)
    _check(conv_state, "conv_state", _conv_state_shape(bsz, dim, width), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    if conv_state_out is None:
        conv_state_out = torch.empty(_conv_state_shape(bsz, dim, width), dtype=torch.float32,
                                     device=dev)
    desc = _b.make_desc(bsz, seqlen, dim, 1, x.dtype, False)
    st = _b.ssm_conv1d_fwd(desc, _b.make_conv_desc(width, activation), x, w, bias, conv_state,
                           out, conv_state_out, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_conv1d_fwd")
    return out, conv_state_out


def conv_scan_fwd(x, conv_w, delta, A, B, C, D=None, z=None, delta_bias=None, conv_bias=None,
                  conv_state=None, initial_state=None, activation=True, delta_softplus=True,
                  out=None, last_state=None, conv_state_out=None, workspace=None, stream=None):
    """The Mamba block's conv + selective scan in one pass: x is the raw
    (pre-conv) input; the scan uses x_conv = act(conv(x) + conv_bias) for both
    the input and the skip term.  Returns ``(out, last_state, conv_state_out)``."""
    if not x.is_cuda:
        raise ValueError("conv_scan_fwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    dstate = A.shape[1]
    width = conv_w.shape[1]
    dev, io = x.device, x.dtype
    _check(delta, "delta", x.shape, io, dev)
    _check(z, "z", x.shape, io, dev)
    _check(B, "B", (bsz, seqlen, dstate), io, dev)
    _check(C, "C", (bsz, seqlen, dstate), io, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _check(initial_state, "initial_state", (bsz, dim, dstate), torch.float32, dev)
    _check(conv_w, "conv_w", (dim, width), torch.float32, dev)
    _check(conv_bias, "conv_bias", (dim,), torch.float32, dev)
    _check(conv_state, "conv_state", _conv_state_shape(bsz, dim, width), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    if last_state is None:
        last_state = torch.empty((bsz, dim, dstate), dtype=torch.float32, device=dev)
    if conv_state_out is None:
        conv_state_out = torch.empty(_conv_state_shape(bsz, dim, width), dtype=torch.float32,
                                     device=dev)
    desc = _b.make_desc(bsz, seqlen, dim, dstate, io, delta_softplus)
    need = _b.ssm_scan_workspace_size(desc)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _b.ssm_conv_scan_fwd(desc, _b.make_conv_desc(width, activation), x, conv_w, conv_bias,
                              conv_state, conv_state_out, delta, A, B, C, D, z, delta_bias, out,
                              last_state, initial_state, workspace if need else None,
                              wbytes if need else 0, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_conv_scan_fwd")
    return out, last_state, conv_state_out


def conv_state_update(conv_state, conv_w, state, x, delta, A, B, C, D=None, z=None,
                      delta_bias=None, conv_bias=None, activation=True, delta_softplus=True,
                      out=None, stream=None):
    """One decode step with the conv in front: conv_state (batch, dim,
    width-1) and state (batch, dim, dstate) are updated in place.  Returns
    ``out``."""
    if not state.is_cuda:
        raise ValueError("conv_state_update runs on a CUDA device only")
    bsz, dim, dstate = state.shape
    width = conv_w.shape[1]
    dev, io = x.device, x.dtype
    _check(state, "state", (bsz, dim, dstate), torch.float32, dev)
    _check(conv_state, "conv_state", _conv_state_shape(bsz, dim, width), torch.float32, dev)
    _check(conv_w, "conv_w", (dim, width), torch.float32, dev)
    _check(conv_bias, "conv_bias", (dim,), torch.float32, dev)
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
    st = _b.ssm_conv_state_update(desc, _b.make_conv_desc(width, activation), conv_state, conv_w,
                                  conv_bias, state, x, delta, A, B, C, D, z, delta_bias, out,
                                  stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_conv_state_update")
    return out


def checkpoint_buffer(x, A):
    """A device buffer for the training forward's checkpoints."""
    bsz, seqlen, dim = x.shape
    desc = _b.make_desc(bsz, seqlen, dim, A.shape[1], x.dtype)
    n = _b.ssm_scan_checkpoint_size(desc) // 4
    return torch.empty(max(n, 4), dtype=torch.float32, device=x.device)


def scan_bwd(x, delta, A, B, C, dout, D=None, z=None, delta_bias=None, initial_state=None,
             dlast_state=None, delta_softplus=True, workspace=None, stream=None, checkpoints=None):
    """Gradients of ``scan_fwd`` for dout = dL/dout (batch, seqlen, dim) and
    optionally dlast_state = dL/dlast_state (batch, dim, dstate) fp32.
    Returns a dict: dx, ddelta, dz (or None without z) in the I/O dtype; dA,
    dB, dC, dD, ddelta_bias, dinitial_state in fp32."""
    if not x.is_cuda:
        raise ValueError("scan_bwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    dstate = A.shape[1]
    dev, io = x.device, x.dtype
    _check(delta, "delta", x.shape, io, dev)
    _check(z, "z", x.shape, io, dev)
    _check(dout, "dout", x.shape, io, dev)
    _check(B, "B", (bsz, seqlen, dstate), io, dev)
    _check(C, "C", (bsz, seqlen, dstate), io, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _check(initial_state, "initial_state", (bsz, dim, dstate), torch.float32, dev)
    _check(dlast_state, "dlast_state", (bsz, dim, dstate), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x),
         "dz": torch.empty_like(x) if z is not None else None,
         "dA": torch.empty((dim, dstate), **f32), "dB": torch.empty((bsz, seqlen, dstate), **f32),
         "dC": torch.empty((bsz, seqlen, dstate), **f32), "dD": torch.empty((dim,), **f32),
         "ddelta_bias": torch.empty((dim,), **f32),
         "dinitial_state": torch.empty((bsz, dim, dstate), **f32)}
    desc = _b.make_desc(bsz, seqlen, dim, dstate, io, delta_softplus)
    need = _b.ssm_scan_bwd_ex_workspace_size(desc, checkpoints is not None)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _b.ssm_scan_bwd_ex(desc, x, delta, A, B, C, D, z, delta_bias, initial_state, dout,
                            dlast_state, checkpoints, g["dx"], g["ddelta"], g["dA"], g["dB"],
                            g["dC"], g["dD"], g["dz"], g["ddelta_bias"], g["dinitial_state"],
                            workspace if need else None, wbytes if need else 0, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_scan_bwd")
    return g


def lti_kernel(delta, A, B, C, seqlen, discretization="euler", stream=None):
    """Convolution kernel (dim, seqlen) fp32 of the time-invariant model:
    delta (dim,), A, B, C (dim, dstate), all fp32 on one device."""
    if not A.is_cuda:
        raise ValueError("lti_kernel runs on a CUDA device only")
    dim, dstate = A.shape
    dev = A.device
    for t, name, shape in ((delta, "delta", (dim,)), (B, "B", (dim, dstate)), (C, "C", (dim, dstate))):
        _check(t, name, shape, torch.float32, dev)
    K = torch.empty((dim, int(seqlen)), dtype=torch.float32, device=dev)
    desc = _b.make_desc(1, seqlen, dim, dstate, torch.float32, False)
    st = _b.ssm_lti_kernel(desc, _b.make_opts(discretization), delta, A, B, C, K, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_lti_kernel")
    return K


def lti_conv_fwd(K, x, D=None, z=None, out=None, stream=None):
    """y = K * x + D x, gated by silu(z): the convolution mode.  K (dim,
    seqlen) fp32; x, z (batch, seqlen, dim)."""
    if not x.is_cuda:
        raise ValueError("lti_conv_fwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    dev, io = x.device, x.dtype
    _check(K, "K", (dim, seqlen), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(z, "z", x.shape, io, dev)
    if out is None:
        out = torch.empty_like(x)
    desc = _b.make_desc(bsz, seqlen, dim, 1, io, False)
    st = _b.ssm_lti_conv_fwd(desc, K, x, D, z, out, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_lti_conv_fwd")
    return out


def selection_proj(x, W_x, W_dt, dt_rank, dstate, delta_bias=None, delta_softplus=False,
                   stream=None):
    """The selection projections: x (batch, seqlen, dim) bf16, W_x (R + 2N,
    dim), W_dt (dim, R) bf16.  Returns ``(dt_low, B, C, delta)``, bf16, shapes
    (batch, seqlen, R | N | N | dim), with delta = act(dt_low W_dt^T +
    delta_bias), act = softplus when ``delta_softplus`` (then delta is the
    step itself: scan it with delta_softplus=False and no bias)."""
    if not x.is_cuda:
        raise ValueError("selection_proj runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    R, N = int(dt_rank), int(dstate)
    dev = x.device
    _check(x, "x", (bsz, seqlen, dim), torch.bfloat16, dev)
    _check(W_x, "W_x", (R + 2 * N, dim), torch.bfloat16, dev)
    _check(W_dt, "W_dt", (dim, R), torch.bfloat16, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    kw = dict(dtype=torch.bfloat16, device=dev)
    dt_low = torch.empty((bsz, seqlen, R), **kw)
    Bm = torch.empty((bsz, seqlen, N), **kw)
    Cm = torch.empty((bsz, seqlen, N), **kw)
    delta = torch.empty((bsz, seqlen, dim), **kw)
    desc = _b.make_desc(bsz, seqlen, dim, N, torch.bfloat16, delta_softplus)
    st = _b.ssm_selection_proj_fwd(desc, _b.ssm_proj_desc(R, 0), x, W_x, W_dt, delta_bias, dt_low,
                                   Bm, Cm, delta, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_selection_proj_fwd")
    return dt_low, Bm, Cm, delta


def proj_scan_fwd(x, dt_low, W_dt, A, B, C, D=None, z=None, delta_bias=None, initial_state=None,
                  out=None, last_state=None, workspace=None, stream=None):
    """The scan with dt_proj fused in front (ssm_proj_scan_fwd): the raw step
    is dt_low W_dt^T, formed inside the scan, then softplus(. + delta_bias).
    x, z: (batch, seqlen, dim) bf16; dt_low (batch, seqlen, R) bf16; W_dt (dim,
    R) bf16; B, C (batch, seqlen, 16) bf16; the rest as scan_fwd.  Returns
    ``(out, last_state)``."""
    if not x.is_cuda:
        raise ValueError("proj_scan_fwd runs on a CUDA device only")
    bsz, seqlen, dim = x.shape
    R = dt_low.shape[-1]
    dstate = A.shape[1]
    dev = x.device
    _check(x, "x", (bsz, seqlen, dim), torch.bfloat16, dev)
    _check(dt_low, "dt_low", (bsz, seqlen, R), torch.bfloat16, dev)
    _check(W_dt, "W_dt", (dim, R), torch.bfloat16, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(B, "B", (bsz, seqlen, dstate), torch.bfloat16, dev)
    _check(C, "C", (bsz, seqlen, dstate), torch.bfloat16, dev)
    _check(z, "z", (bsz, seqlen, dim), torch.bfloat16, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    _check(initial_state, "initial_state", (bsz, dim, dstate), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    if last_state is None:
        last_state = torch.empty((bsz, dim, dstate), dtype=torch.float32, device=dev)
    desc = _b.make_desc(bsz, seqlen, dim, dstate, torch.bfloat16, True)
    need = _b.ssm_scan_workspace_size(desc)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = _b.ssm_proj_scan_fwd(desc, _b.ssm_proj_desc(int(R), 0), x, dt_low, W_dt, A, B, C, D, z,
                              delta_bias, out, last_state, initial_state, workspace,
                              workspace.numel(), stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_proj_scan_fwd")
    return out, last_state


def scan_fwd_host(x, delta, A, B, C, D=None, z=None, delta_bias=None, initial_state=None,
                  delta_softplus=True, slice_batch=0, out=None, last_state=None, workspace=None,
                  stream=None):
    """The scan of host-resident tensors (x, delta, z, B, C, initial_state on
    the CPU, ideally pinned) with A, D, delta_bias on the GPU: slices (whole
    sequences for ``slice_batch`` > 0, runs of -``slice_batch`` steps of one
    sequence for < 0, picked for 0) are copied in, scanned and copied back in
    an overlapped pipeline.  Returns
    ``(out, last_state)`` as CPU tensors (pinned) once the stream reaches the
    end of the call; synchronise the stream before reading them."""
    if x.is_cuda or not A.is_cuda:
        raise ValueError("scan_fwd_host takes host x/delta/z/B/C and device A/D/delta_bias")
    bsz, seqlen, dim = x.shape
    dstate = A.shape[1]
    cpu, dev, io = x.device, A.device, x.dtype
    for t, name, shp in ((delta, "delta", x.shape), (z, "z", x.shape),
                         (B, "B", (bsz, seqlen, dstate)), (C, "C", (bsz, seqlen, dstate))):
        _check(t, name, shp, io, cpu)
    _check(initial_state, "initial_state", (bsz, dim, dstate), torch.float32, cpu)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(D, "D", (dim,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if out is None:
        out = torch.empty(x.shape, dtype=io, pin_memory=True)
    if last_state is None:
        last_state = torch.empty((bsz, dim, dstate), dtype=torch.float32, pin_memory=True)
    desc = _b.make_desc(bsz, seqlen, dim, dstate, io, delta_softplus)
    need = _b.ssm_scan_fwd_host_workspace_size(desc, slice_batch)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=dev)
    ws = workspace
    if ws is not None and ws.data_ptr() % 256:
        off = 256 - ws.data_ptr() % 256
        ws = ws[off:]
    wbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _b.ssm_scan_fwd_host(desc, slice_batch, x, delta, A, B, C, D, z, delta_bias, out,
                              last_state, initial_state, ws if need else None,
                              wbytes if need else 0, stream)
    if st != _b.SSM_OK:
        raise _b.SSMError(st, "ssm_scan_fwd_host")
    return out, last_state
