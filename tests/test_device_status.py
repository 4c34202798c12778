"""Failure detection without a GPU fault: a bounded device-side wait that
runs out sets the library's error word, the kernel returns, the host reads
SSM_ERR_TIMEOUT, the context stays usable, and reading clears the word."""
import time

import pytest
import torch

from parity import TOL, f64, oracle_full, rel_err, to_device
from selective_state_space_137_b300 import binding, ops, synth

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(cuda):
    assert binding.ssm_get_device_status() == binding.SSM_OK
    t0 = time.time()
    assert binding.ssm_selftest_wait_timeout(2_000_000) == binding.SSM_OK     # 2 ms limit
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert binding.ssm_get_device_status() == binding.SSM_ERR_TIMEOUT
    assert binding.ssm_get_device_status() == binding.SSM_OK                  # cleared
    # the context is still usable: a scan right after gives correct results
    w = synth.ScanWorkload("after-timeout", 1, 100, 32, 16, "bf16", 91)
    inp = synth.make_scan_inputs(w)
    out, _ = ops.scan_fwd(**to_device(inp, cuda))
    torch.cuda.synchronize()
    ref, _ = oracle_full(inp)
    assert rel_err(f64(out), ref) <= TOL[torch.bfloat16]
    assert binding.ssm_get_device_status() == binding.SSM_OK


def test_stream_scoped_status(cuda):
    """ssm_get_async_status waits for one stream, then reads and clears the
    same device-wide word."""
    s = torch.cuda.Stream()
    assert binding.ssm_get_async_status(None, s) == binding.SSM_OK
    assert binding.ssm_selftest_wait_timeout(2_000_000, s) == binding.SSM_OK
    assert binding.ssm_get_async_status(None, s) == binding.SSM_ERR_TIMEOUT
    assert binding.ssm_get_async_status(None, s) == binding.SSM_OK     # cleared
    assert binding.ssm_get_device_status() == binding.SSM_OK


def test_selftest_rejects_bad_limits(cuda):
    assert binding.ssm_selftest_wait_timeout(10) == binding.SSM_ERR_INVALID_ARG
    assert binding.ssm_selftest_wait_timeout(10**12) == binding.SSM_ERR_INVALID_ARG
