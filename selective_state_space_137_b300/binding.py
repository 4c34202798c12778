"""ctypes binding of libssm_b300.so: the C ABI of include/ssm.h, one Python
function per entry point with the same name.  This module only marshals
arguments (torch tensors -> device pointers, streams -> handles); every step
of the scan runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssm_b300.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT = 0, 1, 2, 3, 4
SSM_DTYPE_F32, SSM_DTYPE_BF16 = 0, 1

# Every symbol include/ssm.h declares; the CPU tests check the library exports them.
EXPORTED = ("ssm_scan_workspace_size", "ssm_scan_fwd", "ssm_state_update",
            "ssm_scan_plan", "ssm_status_string", "ssm_version", "ssm_scan_fwd_noalloc",
            "ssm_get_device_status", "ssm_get_async_status", "ssm_selftest_wait_timeout", "ssm_conv1d_fwd",
            "ssm_conv_scan_fwd", "ssm_conv_state_update", "ssm_scan_bwd_workspace_size",
            "ssm_scan_bwd", "ssm_scan_fwd_ex", "ssm_state_update_ex", "ssm_lti_kernel",
            "ssm_lti_conv_fwd", "ssm_selection_proj_fwd", "ssm_proj_scan_fwd",
            "ssm_scan_fwd_host_workspace_size",
            "ssm_scan_fwd_host", "ssm_scan_checkpoint_size", "ssm_scan_fwd_train",
            "ssm_scan_bwd_ex_workspace_size", "ssm_scan_bwd_ex", "ssm_scan_bwd_plan")
SSM_DISC_EULER, SSM_DISC_ZOH = 0, 1
SSM_NOALLOC_SCRATCH_BYTES = 8 << 20


class ssm_scan_desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("io_dtype", ctypes.c_int32),
                ("delta_softplus", ctypes.c_int32)]


class ssm_conv_desc(ctypes.Structure):
    _fields_ = [("width", ctypes.c_int32), ("activation", ctypes.c_int32)]


class ssm_scan_opts(ctypes.Structure):
    _fields_ = [("discretization", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


class ssm_proj_desc(ctypes.Structure):
    _fields_ = [("dt_rank", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ssm_scan_plan_info(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("nchunk", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("workspace", ctypes.c_int64)]


class ssm_scan_bwd_plan_info(ctypes.Structure):
    _fields_ = [("nchunk", ctypes.c_int32), ("warps", ctypes.c_int32), ("channels", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("ctas", ctypes.c_int64), ("workspace", ctypes.c_int64)]


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ssm_status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssm_b300.so is not built ({LIB_PATH}); run "
                          "`python -m selective_state_space_137_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, fp, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t
    dp = ctypes.POINTER(ssm_scan_desc)
    lib.ssm_scan_workspace_size.restype = sz
    lib.ssm_scan_workspace_size.argtypes = [dp]
    lib.ssm_scan_fwd.restype = ctypes.c_int
    lib.ssm_scan_fwd.argtypes = [dp, vp, vp, fp, vp, vp, fp, vp, fp, vp, fp, fp, vp, sz, vp]
    lib.ssm_state_update.restype = ctypes.c_int
    lib.ssm_state_update.argtypes = [dp, fp, vp, vp, fp, vp, vp, fp, vp, fp, vp, vp]
    lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
    lib.ssm_scan_fwd_noalloc.argtypes = [dp, vp, vp, fp, vp, vp, fp, vp, fp, vp, fp, fp, vp]
    op = ctypes.POINTER(ssm_scan_opts)
    lib.ssm_scan_fwd_ex.restype = ctypes.c_int
    lib.ssm_scan_fwd_ex.argtypes = [dp, op, vp, vp, fp, vp, vp, fp, vp, fp, vp, fp, fp, vp, sz, vp]
    lib.ssm_state_update_ex.restype = ctypes.c_int
    lib.ssm_state_update_ex.argtypes = [dp, op, fp, vp, vp, fp, vp, vp, fp, vp, fp, vp, vp]
    lib.ssm_lti_kernel.restype = ctypes.c_int
    lib.ssm_lti_kernel.argtypes = [dp, op, fp, fp, fp, fp, fp, vp]
    lib.ssm_lti_conv_fwd.restype = ctypes.c_int
    lib.ssm_lti_conv_fwd.argtypes = [dp, fp, vp, fp, vp, vp, vp]
    lib.ssm_proj_scan_fwd.restype = ctypes.c_int
    lib.ssm_proj_scan_fwd.argtypes = [dp, ctypes.POINTER(ssm_proj_desc), vp, vp, vp, fp, vp, vp, fp,
                                      vp, fp, vp, fp, fp, vp, sz, vp]
    lib.ssm_selection_proj_fwd.restype = ctypes.c_int
    lib.ssm_selection_proj_fwd.argtypes = [dp, ctypes.POINTER(ssm_proj_desc), vp, vp, vp, fp, vp, vp,
                                           vp, vp, vp]
    lib.ssm_scan_fwd_host_workspace_size.restype = sz
    lib.ssm_scan_fwd_host_workspace_size.argtypes = [dp, ctypes.c_int64]
    lib.ssm_scan_fwd_host.restype = ctypes.c_int
    lib.ssm_scan_fwd_host.argtypes = [dp, ctypes.c_int64, vp, vp, fp, vp, vp, fp, vp, fp, vp, fp, fp,
                                      vp, sz, vp]
    lib.ssm_scan_checkpoint_size.restype = sz
    lib.ssm_scan_checkpoint_size.argtypes = [dp]
    lib.ssm_scan_fwd_train.restype = ctypes.c_int
    lib.ssm_scan_fwd_train.argtypes = [dp, vp, vp, fp, vp, vp, fp, vp, fp, vp, fp, fp, fp, vp, sz, vp]
    lib.ssm_scan_bwd_ex_workspace_size.restype = sz
    lib.ssm_scan_bwd_ex_workspace_size.argtypes = [dp, ctypes.c_int]
    lib.ssm_scan_bwd_ex.restype = ctypes.c_int
    lib.ssm_scan_bwd_ex.argtypes = [dp, vp, vp, fp, vp, vp, fp, vp, fp, fp, vp, fp, fp, vp, vp, fp, fp,
                                    fp, fp, vp, fp, fp, vp, sz, vp]
    lib.ssm_scan_bwd_workspace_size.restype = sz
    lib.ssm_scan_bwd_workspace_size.argtypes = [dp]
    lib.ssm_scan_bwd.restype = ctypes.c_int
    lib.ssm_scan_bwd.argtypes = [dp, vp, vp, fp, vp, vp, fp, vp, fp, fp, vp, fp, vp, vp, fp, fp, fp,
                                 fp, vp, fp, fp, vp, sz, vp]
    cp = ctypes.POINTER(ssm_conv_desc)
    lib.ssm_conv1d_fwd.restype = ctypes.c_int
    lib.ssm_conv1d_fwd.argtypes = [dp, cp, vp, fp, fp, fp, vp, fp, vp]
    lib.ssm_conv_scan_fwd.restype = ctypes.c_int
    lib.ssm_conv_scan_fwd.argtypes = [dp, cp, vp, fp, fp, fp, fp, vp, fp, vp, vp, fp, vp, fp, vp,
                                      fp, fp, vp, sz, vp]
    lib.ssm_conv_state_update.restype = ctypes.c_int
    lib.ssm_conv_state_update.argtypes = [dp, cp, fp, fp, fp, fp, vp, vp, fp, vp, vp, fp, vp, fp,
                                          vp, vp]
    lib.ssm_scan_plan.restype = ctypes.c_int
    lib.ssm_scan_plan.argtypes = [dp, ctypes.POINTER(ssm_scan_plan_info)]
    lib.ssm_scan_bwd_plan.restype = ctypes.c_int
    lib.ssm_scan_bwd_plan.argtypes = [dp, ctypes.c_int, ctypes.POINTER(ssm_scan_bwd_plan_info)]
    lib.ssm_selftest_wait_timeout.restype = ctypes.c_int
    lib.ssm_selftest_wait_timeout.argtypes = [ctypes.c_int64, vp]
    lib.ssm_get_device_status.restype = ctypes.c_int
    lib.ssm_get_device_status.argtypes = []
    lib.ssm_get_async_status.restype = ctypes.c_int
    lib.ssm_get_async_status.argtypes = [vp, vp]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [ctypes.c_int]
    lib.ssm_version.restype = ctypes.c_int
    lib.ssm_version.argtypes = []
    return lib


lib = _load()


def ssm_status_string(status: int) -> str:
    return lib.ssm_status_string(int(status)).decode()


def ssm_get_device_status() -> int:
    return lib.ssm_get_device_status()


def ssm_get_async_status(workspace=None, stream=None) -> int:
    return lib.ssm_get_async_status(_ptr(workspace), _stream(stream))


def ssm_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return lib.ssm_selftest_wait_timeout(int(limit_ns), _stream(stream))


def ssm_version() -> int:
    return lib.ssm_version()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _io_code(dtype) -> int:
    if dtype == torch.float32:
        return SSM_DTYPE_F32
    if dtype == torch.bfloat16:
        return SSM_DTYPE_BF16
    raise TypeError(f"unsupported io dtype {dtype}")


def make_desc(batch, seqlen, dim, dstate, io_dtype, delta_softplus=True) -> ssm_scan_desc:
    io = io_dtype if isinstance(io_dtype, int) else _io_code(io_dtype)
    return ssm_scan_desc(int(batch), int(seqlen), int(dim), int(dstate), io,
                         1 if delta_softplus else 0)


def ssm_scan_workspace_size(desc: ssm_scan_desc) -> int:
    return int(lib.ssm_scan_workspace_size(ctypes.byref(desc)))


def ssm_scan_plan(desc: ssm_scan_desc) -> ssm_scan_plan_info:
    info = ssm_scan_plan_info()
    st = lib.ssm_scan_plan(ctypes.byref(desc), ctypes.byref(info))
    if st != SSM_OK:
        raise SSMError(st, "ssm_scan_plan")
    return info


def ssm_scan_bwd_plan(desc: ssm_scan_desc, with_checkpoints: bool = False) -> ssm_scan_bwd_plan_info:
    info = ssm_scan_bwd_plan_info()
    st = lib.ssm_scan_bwd_plan(ctypes.byref(desc), int(bool(with_checkpoints)), ctypes.byref(info))
    if st != SSM_OK:
        raise SSMError(st, "ssm_scan_bwd_plan")
    return info


def ssm_scan_fwd(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state, initial_state,
                 workspace, workspace_bytes, stream=None) -> int:
    """Direct call of the C entry point; tensors (or raw device addresses) in,
    status code out."""
    return lib.ssm_scan_fwd(ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                            _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out), _ptr(last_state),
                            _ptr(initial_state), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def ssm_state_update(desc, state, x, delta, A, B, C, D, z, delta_bias, out, stream=None) -> int:
    return lib.ssm_state_update(ctypes.byref(desc), _ptr(state), _ptr(x), _ptr(delta), _ptr(A),
                                _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out),
                                _stream(stream))


def ssm_scan_fwd_noalloc(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                         initial_state, stream=None) -> int:
    """The scan for callers that cannot allocate: no workspace argument; the
    library's fixed device scratch array is used instead."""
    return lib.ssm_scan_fwd_noalloc(ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(B),
                                    _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out),
                                    _ptr(last_state), _ptr(initial_state), _stream(stream))


def make_conv_desc(width, activation=True) -> ssm_conv_desc:
    return ssm_conv_desc(int(width), 1 if activation else 0)


def ssm_conv1d_fwd(desc, conv, x, w, bias, conv_state_in, out, conv_state_out, stream=None) -> int:
    """Causal depthwise conv (+ SiLU) of x, standalone; status code out."""
    return lib.ssm_conv1d_fwd(ctypes.byref(desc), ctypes.byref(conv), _ptr(x), _ptr(w), _ptr(bias),
                              _ptr(conv_state_in), _ptr(out), _ptr(conv_state_out), _stream(stream))


def ssm_conv_scan_fwd(desc, conv, x, conv_w, conv_bias, conv_state_in, conv_state_out, delta, A,
                      B, C, D, z, delta_bias, out, last_state, initial_state, workspace,
                      workspace_bytes, stream=None) -> int:
    """The conv fused in front of the scan (x is the raw, pre-conv input)."""
    return lib.ssm_conv_scan_fwd(ctypes.byref(desc), ctypes.byref(conv), _ptr(x), _ptr(conv_w),
                                 _ptr(conv_bias), _ptr(conv_state_in), _ptr(conv_state_out),
                                 _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                 _ptr(delta_bias), _ptr(out), _ptr(last_state),
                                 _ptr(initial_state), _ptr(workspace), int(workspace_bytes),
                                 _stream(stream))


def ssm_conv_state_update(desc, conv, conv_state, conv_w, conv_bias, state, x, delta, A, B, C, D,
                          z, delta_bias, out, stream=None) -> int:
    """One decode step with the conv in front; conv_state and state in place."""
    return lib.ssm_conv_state_update(ctypes.byref(desc), ctypes.byref(conv), _ptr(conv_state),
                                     _ptr(conv_w), _ptr(conv_bias), _ptr(state), _ptr(x),
                                     _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                     _ptr(delta_bias), _ptr(out), _stream(stream))


def ssm_scan_bwd_workspace_size(desc: ssm_scan_desc) -> int:
    return int(lib.ssm_scan_bwd_workspace_size(ctypes.byref(desc)))


def ssm_scan_bwd(desc, x, delta, A, B, C, D, z, delta_bias, initial_state, dout, dlast_state, dx,
                 ddelta, dA, dB, dC, dD, dz, ddelta_bias, dinitial_state, workspace,
                 workspace_bytes, stream=None) -> int:
    """Gradients of the scan (the states are recomputed); status code out."""
    return lib.ssm_scan_bwd(ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                            _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(initial_state), _ptr(dout),
                            _ptr(dlast_state), _ptr(dx), _ptr(ddelta), _ptr(dA), _ptr(dB),
                            _ptr(dC), _ptr(dD), _ptr(dz), _ptr(ddelta_bias),
                            _ptr(dinitial_state), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def make_opts(discretization="euler") -> ssm_scan_opts:
    code = {"euler": SSM_DISC_EULER, "zoh": SSM_DISC_ZOH}.get(discretization, discretization)
    o = ssm_scan_opts()
    o.discretization = int(code)
    return o


def ssm_scan_fwd_ex(desc, opts, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                    initial_state, workspace, workspace_bytes, stream=None) -> int:
    """ssm_scan_fwd with options (opts: ssm_scan_opts or None)."""
    return lib.ssm_scan_fwd_ex(ctypes.byref(desc), None if opts is None else ctypes.byref(opts),
                               _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                               _ptr(delta_bias), _ptr(out), _ptr(last_state),
                               _ptr(initial_state), _ptr(workspace), int(workspace_bytes),
                               _stream(stream))


def ssm_state_update_ex(desc, opts, state, x, delta, A, B, C, D, z, delta_bias, out,
                        stream=None) -> int:
    return lib.ssm_state_update_ex(ctypes.byref(desc), None if opts is None else ctypes.byref(opts),
                                   _ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                   _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out), _stream(stream))


def ssm_lti_kernel(desc, opts, delta, A, B, C, K, stream=None) -> int:
    """Convolution kernel K (dim, seqlen) of the time-invariant model."""
    return lib.ssm_lti_kernel(ctypes.byref(desc), None if opts is None else ctypes.byref(opts),
                              _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(K), _stream(stream))


def ssm_lti_conv_fwd(desc, K, x, D, z, out, stream=None) -> int:
    """y = K * x + D x (gated by silu(z)), the convolution mode."""
    return lib.ssm_lti_conv_fwd(ctypes.byref(desc), _ptr(K), _ptr(x), _ptr(D), _ptr(z), _ptr(out),
                                _stream(stream))


def ssm_proj_scan_fwd(desc, proj, x, dt_low, W_dt, A, B, C, D, z, delta_bias, out, last_state,
                      initial_state, workspace, workspace_bytes, stream=None):
    return lib.ssm_proj_scan_fwd(ctypes.byref(desc), ctypes.byref(proj), _ptr(x), _ptr(dt_low),
                                 _ptr(W_dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                 _ptr(delta_bias), _ptr(out), _ptr(last_state), _ptr(initial_state),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream))


def ssm_selection_proj_fwd(desc, proj, x, W_x, W_dt, delta_bias, dt_low, B, C, delta,
                           stream=None) -> int:
    """x_proj (-> dt_low, B, C) and dt_proj (-> delta = act(dt_low W_dt^T +
    delta_bias), act = softplus iff desc.delta_softplus) on the tensor cores."""
    return lib.ssm_selection_proj_fwd(ctypes.byref(desc), ctypes.byref(proj), _ptr(x), _ptr(W_x),
                                      _ptr(W_dt), _ptr(delta_bias), _ptr(dt_low), _ptr(B), _ptr(C),
                                      _ptr(delta), _stream(stream))


def ssm_scan_fwd_host_workspace_size(desc, slice_batch=0) -> int:
    return int(lib.ssm_scan_fwd_host_workspace_size(ctypes.byref(desc), int(slice_batch)))


def ssm_scan_fwd_host(desc, slice_batch, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                      initial_state, workspace, workspace_bytes, stream=None) -> int:
    """The scan over host tensors (x, delta, z, B, C, out, states: host
    memory, pinned for overlap; A, D, delta_bias: device), pipelined over
    slices through a device workspace (slice_batch > 0: whole sequences,
    < 0: runs of that many steps of one sequence, 0: picked)."""
    return lib.ssm_scan_fwd_host(ctypes.byref(desc), int(slice_batch), _ptr(x), _ptr(delta), _ptr(A),
                                 _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out),
                                 _ptr(last_state), _ptr(initial_state), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))


def ssm_scan_checkpoint_size(desc) -> int:
    return int(lib.ssm_scan_checkpoint_size(ctypes.byref(desc)))


def ssm_scan_fwd_train(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state, initial_state,
                       checkpoints, workspace, workspace_bytes, stream=None) -> int:
    """ssm_scan_fwd that also keeps the state before every 16th token."""
    return lib.ssm_scan_fwd_train(ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(B),
                                  _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(out),
                                  _ptr(last_state), _ptr(initial_state), _ptr(checkpoints),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream))


def ssm_scan_bwd_ex_workspace_size(desc, with_checkpoints) -> int:
    return int(lib.ssm_scan_bwd_ex_workspace_size(ctypes.byref(desc), int(bool(with_checkpoints))))


def ssm_scan_bwd_ex(desc, x, delta, A, B, C, D, z, delta_bias, initial_state, dout, dlast_state,
                    checkpoints, dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dinitial_state,
                    workspace, workspace_bytes, stream=None) -> int:
    """ssm_scan_bwd reading the forward's checkpoints (NULL: recompute)."""
    return lib.ssm_scan_bwd_ex(ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(initial_state), _ptr(dout),
                               _ptr(dlast_state), _ptr(checkpoints), _ptr(dx), _ptr(ddelta),
                               _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD), _ptr(dz),
                               _ptr(ddelta_bias), _ptr(dinitial_state), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))
