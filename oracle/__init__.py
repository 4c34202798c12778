"""fp64 CPU oracle for the selective state-space scan (S6).

TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything here, and nothing here imports the CUDA
library: the two share only the seeded input generator, which holds none of
the method's arithmetic.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, libm ``exp`` and
``log1p``), compiled on first use into ``liboracle.so`` next to this file.
This module only marshals numpy arrays into fp64 buffers for it.

Definitions followed (see the header of ``ssm_oracle.c`` for the passages):
the recurrence h_t = exp(Delta_t A) * h_{t-1} + Delta_t B_t x_t, the readout
y_t = C_t . h_t + D x_t, the gate silu(z_t), and Delta = softplus(raw + bias);
the causal depthwise conv in front of it; the gradients of the scan
(``scan_bwd``: the same loop differentiated in reverse mode); the exact
zero-order-hold input term (``scan_fwd(zoh=True)``); and the time-invariant
convolution mode (``lti_kernel``, ``lti_conv``).

Every function here is pinned by ``tests/test_oracle_pins.py`` against
identities and closed forms that are independent of this code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (fp64, no fast-math, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def build_variant(out_path: str, source_text: str) -> str:
    """Compile an edited copy of the oracle source (used by the mutation
    tests, which plant a mistake in a copy to show the pins catch it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
                    "-fPIC", "-shared", "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib):
    lib.oracle_scan_fwd.restype = ctypes.c_int
    lib.oracle_scan_fwd.argtypes = [ctypes.c_int64] * 4 + [_dp] * 8 + [ctypes.c_int, _dp, _dp, _dp,
                                                                       ctypes.c_int]
    lib.oracle_state_update.restype = ctypes.c_int
    lib.oracle_state_update.argtypes = [ctypes.c_int64] * 3 + [_dp] * 9 + [ctypes.c_int, _dp]
    lib.oracle_scan_fwd_zoh.restype = ctypes.c_int
    lib.oracle_scan_fwd_zoh.argtypes = lib.oracle_scan_fwd.argtypes
    lib.oracle_lti_kernel.restype = ctypes.c_int
    lib.oracle_lti_kernel.argtypes = [ctypes.c_int64] * 3 + [_dp] * 4 + [ctypes.c_int, _dp]
    lib.oracle_lti_conv.restype = ctypes.c_int
    lib.oracle_lti_conv.argtypes = [ctypes.c_int64] * 3 + [_dp] * 5
    lib.oracle_scan_bwd.restype = ctypes.c_int
    lib.oracle_scan_bwd.argtypes = ([ctypes.c_int64] * 4 + [_dp] * 8 + [ctypes.c_int] + [_dp] * 12
                                    + [ctypes.c_int])
    lib.oracle_conv1d_fwd.restype = ctypes.c_int
    lib.oracle_conv1d_fwd.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] + [_dp] * 6
    lib.oracle_softplus_scalar.restype = ctypes.c_double
    lib.oracle_softplus_scalar.argtypes = [ctypes.c_double]
    lib.oracle_silu_scalar.restype = ctypes.c_double
    lib.oracle_silu_scalar.argtypes = [ctypes.c_double]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` selects a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(a, shape=None):
    if a is None:
        return None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and arr.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {arr.shape}")
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
             initial_state=None, nthreads=0, lib=None, zoh=False):
    """Selective scan forward in fp64.

    x, delta, z: (batch, seqlen, dim); B, C: (batch, seqlen, dstate);
    A: (dim, dstate); D, delta_bias: (dim,); initial_state: (batch, dim, dstate).
    Returns ``(out, last_state)``, fp64 arrays of shapes (batch, seqlen, dim) and
    (batch, dim, dstate).  ``zoh=True`` takes the exact zero-order-hold input
    term ((exp(Delta A) - 1) / A) B x instead of Delta B x.
    """
    x = _f64(x)
    bsz, seqlen, dim = x.shape
    A = _f64(A)
    dstate = A.shape[1]
    delta = _f64(delta, x.shape)
    B = _f64(B, (bsz, seqlen, dstate))
    C = _f64(C, (bsz, seqlen, dstate))
    D = _f64(D, (dim,))
    z = _f64(z, x.shape)
    delta_bias = _f64(delta_bias, (dim,))
    initial_state = _f64(initial_state, (bsz, dim, dstate))
    out = np.empty((bsz, seqlen, dim), dtype=np.float64)
    last = np.empty((bsz, dim, dstate), dtype=np.float64)
    L_ = lib or load()
    fn = L_.oracle_scan_fwd_zoh if zoh else L_.oracle_scan_fwd
    rc = fn(bsz, seqlen, dim, dstate, _ptr(x), _ptr(delta), _ptr(A),
                                         _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                         int(bool(delta_softplus)), _ptr(initial_state), _ptr(out),
                                         _ptr(last), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_scan_fwd rejected its arguments")
    return out, last


def scan_bwd(x, delta, A, B, C, dout, D=None, z=None, delta_bias=None, delta_softplus=True,
             initial_state=None, dlast_state=None, nthreads=0, lib=None):
    """Gradients of ``scan_fwd`` in fp64, given dout = dL/dout (batch, seqlen,
    dim) and optionally dlast_state = dL/dlast_state (batch, dim, dstate).
    Returns a dict with dx, ddelta, dA, dB, dC, dD, dz (None without z),
    ddelta_bias and dinitial_state (gradients w.r.t. D, the bias and the
    initial state are returned whether or not those inputs were given: they
    are the gradients at zero)."""
    x = _f64(x)
    bsz, seqlen, dim = x.shape
    A = _f64(A)
    dstate = A.shape[1]
    delta = _f64(delta, x.shape)
    B = _f64(B, (bsz, seqlen, dstate))
    C = _f64(C, (bsz, seqlen, dstate))
    D = _f64(D, (dim,))
    z = _f64(z, x.shape)
    delta_bias = _f64(delta_bias, (dim,))
    initial_state = _f64(initial_state, (bsz, dim, dstate))
    dout = _f64(dout, x.shape)
    dlast_state = _f64(dlast_state, (bsz, dim, dstate))
    g = {k: np.empty(sh, dtype=np.float64) for k, sh in (
        ("dx", x.shape), ("ddelta", x.shape), ("dA", (dim, dstate)), ("dB", B.shape),
        ("dC", C.shape), ("dD", (dim,)), ("ddelta_bias", (dim,)),
        ("dinitial_state", (bsz, dim, dstate)))}
    g["dz"] = np.empty(x.shape, dtype=np.float64) if z is not None else None
    rc = (lib or load()).oracle_scan_bwd(
        bsz, seqlen, dim, dstate, _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(initial_state), _ptr(dout),
        _ptr(dlast_state), _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]),
        _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]),
        _ptr(g["dinitial_state"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_scan_bwd rejected its arguments")
    return g


def state_update(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 lib=None):
    """One decode step in fp64.  ``state`` (batch, dim, dstate) is not modified;
    the updated state is returned with the output: ``(out, new_state)``."""
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    bsz, dim, dstate = st.shape
    x = _f64(x, (bsz, dim))
    delta = _f64(delta, (bsz, dim))
    A = _f64(A, (dim, dstate))
    B = _f64(B, (bsz, dstate))
    C = _f64(C, (bsz, dstate))
    D = _f64(D, (dim,))
    z = _f64(z, (bsz, dim))
    delta_bias = _f64(delta_bias, (dim,))
    out = np.empty((bsz, dim), dtype=np.float64)
    rc = (lib or load()).oracle_state_update(bsz, dim, dstate, _ptr(st), _ptr(x), _ptr(delta),
                                             _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                             _ptr(delta_bias), int(bool(delta_softplus)),
                                             _ptr(out))
    if rc != 0:
        raise ValueError("oracle_state_update rejected its arguments")
    return out, st


def lti_kernel(delta, A, B, C, seqlen, zoh=False, lib=None):
    """Convolution kernel K (dim, seqlen) of the time-invariant model with
    per-channel step delta (dim,) and per-channel B, C (dim, dstate)."""
    A = _f64(A)
    dim, dstate = A.shape
    delta = _f64(delta, (dim,))
    B = _f64(B, (dim, dstate))
    C = _f64(C, (dim, dstate))
    K = np.empty((dim, int(seqlen)), dtype=np.float64)
    rc = (lib or load()).oracle_lti_kernel(dim, dstate, int(seqlen), _ptr(delta), _ptr(A), _ptr(B),
                                           _ptr(C), int(bool(zoh)), _ptr(K))
    if rc != 0:
        raise ValueError("oracle_lti_kernel rejected its arguments")
    return K


def lti_conv(K, x, D=None, z=None, lib=None):
    """y = K * x (causal, per channel) + D x, gated by silu(z) when given.
    K: (dim, seqlen); x, z: (batch, seqlen, dim)."""
    x = _f64(x)
    bsz, seqlen, dim = x.shape
    K = _f64(K, (dim, seqlen))
    D = _f64(D, (dim,))
    z = _f64(z, x.shape)
    out = np.empty(x.shape, dtype=np.float64)
    rc = (lib or load()).oracle_lti_conv(bsz, seqlen, dim, _ptr(K), _ptr(x), _ptr(D), _ptr(z),
                                         _ptr(out))
    if rc != 0:
        raise ValueError("oracle_lti_conv rejected its arguments")
    return out


def selection_proj(x, W_x, W_dt, dt_rank):
    """The input-dependent selection of S6 ("Mamba的三大创新", the selection
    mechanism: Delta, B and C computed from the input by linear projections):
        xdbl = x W_x^T                  (tokens, dt_rank + 2 N)
        dt_low, B, C = xdbl[:, :R], xdbl[:, R:R+N], xdbl[:, R+N:]
        delta_raw = dt_low W_dt^T       (tokens, dim)
    x: (batch, seqlen, dim); W_x: (R + 2N, dim); W_dt: (dim, R).  fp64 numpy
    matmuls (a library primitive as the step).  Returns (dt_low, B, C,
    delta_raw) with the leading (batch, seqlen) shape."""
    x = _f64(x)
    W_x = _f64(W_x)
    W_dt = _f64(W_dt)
    bsz, seqlen, dim = x.shape
    R = int(dt_rank)
    N2 = W_x.shape[0] - R
    if W_x.shape[1] != dim or W_dt.shape != (dim, R) or N2 <= 0 or N2 % 2:
        raise ValueError("W_x must be (R + 2N, dim) and W_dt (dim, R)")
    xdbl = x.reshape(-1, dim) @ W_x.T
    dt_low = xdbl[:, :R]
    N = N2 // 2
    Bm = xdbl[:, R:R + N]
    Cm = xdbl[:, R + N:]
    shp = (bsz, seqlen)
    dt_low = dt_low.reshape(*shp, R)
    return dt_low, Bm.reshape(*shp, N), Cm.reshape(*shp, N), dt_proj(dt_low, W_dt)


def dt_proj(dt_low, W_dt):
    """The second selection projection alone: delta_raw = dt_low W_dt^T, the
    raw step of every token and channel.  dt_low: (batch, seqlen, R); W_dt:
    (dim, R).  fp64 numpy matmul.  Returns (batch, seqlen, dim)."""
    dt_low = _f64(dt_low)
    W_dt = _f64(W_dt)
    if dt_low.ndim != 3 or W_dt.ndim != 2 or W_dt.shape[1] != dt_low.shape[2]:
        raise ValueError("dt_low must be (batch, seqlen, R) and W_dt (dim, R)")
    return dt_low @ W_dt.T


def conv1d_fwd(x, w, bias=None, conv_state=None, activation=True, lib=None):
    """Causal depthwise conv1d (+ SiLU) in fp64.  x: (batch, seqlen, dim);
    w: (dim, width); bias: (dim,); conv_state: (batch, dim, width-1) inputs
    before t = 0 (oldest first) or None for zeros.
    Returns ``(out, conv_state_out)``."""
    x = _f64(x)
    bsz, seqlen, dim = x.shape
    w = _f64(w)
    width = w.shape[1]
    if w.shape[0] != dim:
        raise ValueError("w must be (dim, width)")
    bias = _f64(bias, (dim,))
    conv_state = _f64(conv_state, (bsz, dim, width - 1))
    out = np.empty((bsz, seqlen, dim), dtype=np.float64)
    st = np.empty((bsz, dim, width - 1), dtype=np.float64)
    rc = (lib or load()).oracle_conv1d_fwd(bsz, seqlen, dim, width, int(bool(activation)),
                                           _ptr(x), _ptr(w), _ptr(bias), _ptr(conv_state),
                                           _ptr(out), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_conv1d_fwd rejected its arguments")
    return out, st


def softplus(u: float, lib=None) -> float:
    return (lib or load()).oracle_softplus_scalar(float(u))


def silu(v: float, lib=None) -> float:
    return (lib or load()).oracle_silu_scalar(float(v))
