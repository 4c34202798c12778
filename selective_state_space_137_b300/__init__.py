"""B300-native selective state-space scan (Mamba S6).

Prefill (``scan_fwd``), its gradients (``scan_bwd``), decode
(``state_update``), and prefill and decode with
the Mamba block's causal conv fused in front (``conv_scan_fwd``,
``conv_state_update``; ``conv1d_fwd`` is the conv alone), run in hand-written
CUDA kernels for sm_103a behind the C ABI of ``include/ssm.h``
(libssm_b300.so).
PyTorch supplies device memory and streams only.

The CUDA library is loaded on first use of an op: importing the package
itself (e.g. for ``synth``) does not need it, but any op raises if the
library is missing -- there is no CPU fallback.
"""
from __future__ import annotations

import importlib

_OPS = ("scan_fwd", "scan_bwd", "state_update", "conv1d_fwd", "conv_scan_fwd",
        "conv_state_update", "lti_kernel", "lti_conv_fwd", "selection_proj", "scan_fwd_host")
__all__ = list(_OPS) + ["binding", "synth", "ops"]


def __getattr__(name):
    if name in _OPS:
        return getattr(importlib.import_module(__name__ + ".ops"), name)
    if name in ("binding", "synth", "ops"):
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
