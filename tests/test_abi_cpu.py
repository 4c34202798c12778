"""The C ABI without a GPU: the library loads, exports every symbol that
include/ssm.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("ssm_scan_fwd", "ssm_state_update", "ssm_scan_workspace_size",
              "ssm_status_string", "ssm_version"):
        assert n in names


def test_library_exports_every_declared_symbol(ssm_lib):
    lib = ctypes.CDLL(ssm_lib.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(declared_symbols()) <= set(ssm_lib.EXPORTED) | set(declared_symbols())


def test_status_strings_and_version(ssm_lib):
    for code in range(5):
        assert ssm_lib.ssm_status_string(code).startswith("SSM_")
    assert "unknown" in ssm_lib.ssm_status_string(99)
    assert ssm_lib.ssm_version() >= 100


def test_workspace_size(ssm_lib):
    d = ssm_lib.make_desc(4, 8192, 4096, 16, ssm_lib.SSM_DTYPE_BF16)
    assert ssm_lib.ssm_scan_workspace_size(d) % 4 == 0
    long = ssm_lib.make_desc(1, 262144, 2048, 16, ssm_lib.SSM_DTYPE_BF16)
    assert ssm_lib.ssm_scan_workspace_size(long) > 0     # long sequence, few channels: chunked
    bad = ssm_lib.make_desc(1, 16, 16, 3, ssm_lib.SSM_DTYPE_F32)
    assert ssm_lib.ssm_scan_workspace_size(bad) == 0
    assert ssm_lib.lib.ssm_scan_workspace_size(None) == 0


# Fake, never-dereferenced addresses: every call below must return before any CUDA work.
A16 = 0x10000


def _scan(ssm_lib, desc, x=A16, ws=None, wsb=0, misalign=0):
    return ssm_lib.ssm_scan_fwd(desc, x + misalign, A16, A16, A16, A16, None, None, None, A16,
                                None, None, ws, wsb, None)


def test_rejections_before_launch(ssm_lib):
    L = ssm_lib
    good = L.make_desc(1, 8, 16, 4, L.SSM_DTYPE_F32)
    assert L.lib.ssm_scan_fwd(None, *([None] * 11), None, 0, None) == L.SSM_ERR_INVALID_ARG
    assert _scan(L, L.make_desc(-1, 8, 16, 4, 0)) == L.SSM_ERR_INVALID_ARG
    assert _scan(L, L.make_desc(1, 8, 16, 3, 0)) == L.SSM_ERR_UNSUPPORTED
    assert _scan(L, L.make_desc(1, 8, 16, 128, 0)) == L.SSM_ERR_UNSUPPORTED
    assert _scan(L, L.make_desc(1, 8, 16, 4, 7)) == L.SSM_ERR_UNSUPPORTED
    assert _scan(L, good, misalign=2) == L.SSM_ERR_INVALID_ARG           # fp32 at a 2-byte offset
    assert _scan(L, L.make_desc(1, 8, 16, 4, L.SSM_DTYPE_BF16), misalign=1) == L.SSM_ERR_INVALID_ARG
    assert _scan(L, good, x=0) == L.SSM_ERR_INVALID_ARG                  # NULL x
    assert _scan(L, L.make_desc(0, 8, 16, 4, 0)) == L.SSM_OK              # empty batch: no-op
    long = L.make_desc(1, 262144, 2048, 16, L.SSM_DTYPE_BF16)
    need = L.ssm_scan_plan(long).workspace        # the path these aligned addresses take
    assert 0 < need <= L.ssm_scan_workspace_size(long)
    assert _scan(L, long, ws=None, wsb=0) == L.SSM_ERR_INVALID_ARG        # workspace missing
    assert _scan(L, long, ws=A16, wsb=need - 16) == L.SSM_ERR_INVALID_ARG  # too small
    assert L.ssm_state_update(good, A16 + 8, A16, A16, A16, A16, A16, None, None, None, A16) \
        == L.SSM_ERR_INVALID_ARG
    assert L.ssm_state_update(L.make_desc(1, 1, 16, 5, 0), A16, A16, A16, A16, A16, A16, None,
                              None, None, A16) == L.SSM_ERR_UNSUPPORTED


def test_ops_refuse_cpu_tensors(ssm_lib):
    from selective_state_space_137_b300 import ops
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        ops.scan_fwd(x, x, torch.zeros(8, 4), torch.zeros(1, 4, 4), torch.zeros(1, 4, 4))
    with pytest.raises(ValueError):
        ops.state_update(torch.zeros(1, 8, 4), x[:, 0], x[:, 0], torch.zeros(8, 4),
                         torch.zeros(1, 4), torch.zeros(1, 4))


def test_synthetic_inputs_are_seeded():
    from selective_state_space_137_b300 import synth
    a = synth.make_scan_inputs(synth.TINY)
    b = synth.make_scan_inputs(synth.TINY)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k])
    assert a["x"].dtype == torch.float32 and a["A"][0, 3].item() == -4.0
    bias = a["delta_bias"].double()
    dt = torch.nn.functional.softplus(bias)
    assert torch.all(dt > 1e-3 * 0.999) and torch.all(dt < 0.1 * 1.001)


def test_plan_picks_the_tiled_path(ssm_lib):
    L = ssm_lib
    big = L.ssm_scan_plan(L.make_desc(4, 8192, 4096, 16, L.SSM_DTYPE_BF16))
    assert (big.path, big.nchunk, big.launches, big.workspace) == (3, 1, 1, 0)
    long = L.ssm_scan_plan(L.make_desc(1, 262144, 2048, 16, L.SSM_DTYPE_BF16))
    assert long.path == 3 and long.nchunk > 1 and long.launches == 3 and long.workspace > 0
    # one wave of one-warp CTAs: 128 channel groups x chunks <= 148 SMs x 8
    assert 8 <= long.nchunk and long.nchunk * 128 <= 148 * 8
    assert L.ssm_scan_workspace_size(L.make_desc(1, 262144, 2048, 16, L.SSM_DTYPE_BF16)) >= long.workspace
    for n, path in ((1, 0), (2, 0), (4, 0), (8, 3), (16, 3), (32, 3), (64, 3)):
        assert L.ssm_scan_plan(L.make_desc(2, 300, 72, n, L.SSM_DTYPE_BF16)).path == path
    assert L.ssm_scan_plan(L.make_desc(2, 300, 72, 16, L.SSM_DTYPE_F32)).path == 3
    assert L.ssm_scan_plan(L.make_desc(2, 300, 12, 16, L.SSM_DTYPE_BF16)).path == 0   # 24-byte rows


def test_conv_rejections_before_launch(ssm_lib):
    """The conv entry points check the conv descriptor, alignment and aliasing
    before any CUDA call (fake addresses again)."""
    L = ssm_lib
    d = L.make_desc(2, 8, 16, 16, L.SSM_DTYPE_F32)
    ok_conv = L.make_conv_desc(4, True)

    def conv1d(conv, x=A16, w=A16, s_in=None, out=A16 + 4096, s_out=None, desc=d):
        return L.ssm_conv1d_fwd(desc, conv, x, w, None, s_in, out, s_out, None)

    assert L.lib.ssm_conv1d_fwd(ctypes.byref(d), None, *([None] * 7)) == L.SSM_ERR_INVALID_ARG
    assert conv1d(L.make_conv_desc(0)) == L.SSM_ERR_UNSUPPORTED            # width 0
    assert conv1d(L.make_conv_desc(9)) == L.SSM_ERR_UNSUPPORTED            # width > 8
    assert conv1d(L.ssm_conv_desc(4, 2)) == L.SSM_ERR_INVALID_ARG          # activation not 0/1
    assert conv1d(ok_conv, x=A16 + 2) == L.SSM_ERR_INVALID_ARG             # fp32 at 2-byte offset
    assert conv1d(ok_conv, s_in=A16, s_out=A16 + 8) == L.SSM_ERR_INVALID_ARG   # states overlap
    assert conv1d(ok_conv, x=0) == L.SSM_ERR_INVALID_ARG                   # NULL x
    assert conv1d(ok_conv, out=A16 + 64) == L.SSM_ERR_INVALID_ARG          # out overlaps x
    assert conv1d(ok_conv, desc=L.make_desc(0, 8, 16, 1, 0)) == L.SSM_OK   # empty batch: no-op

    def fused(conv, w=A16, s_in=None, s_out=None, desc=d):
        return L.ssm_conv_scan_fwd(desc, conv, A16, w, None, s_in, s_out, A16, A16, A16, A16,
                                   None, None, None, A16, None, None, None, 0, None)

    assert fused(L.make_conv_desc(9)) == L.SSM_ERR_UNSUPPORTED
    assert fused(ok_conv, w=0) == L.SSM_ERR_INVALID_ARG                    # taps missing
    assert fused(ok_conv, s_in=A16, s_out=A16) == L.SSM_ERR_INVALID_ARG    # in-place conv state
    assert fused(ok_conv, desc=L.make_desc(1, 8, 16, 3, 0)) == L.SSM_ERR_UNSUPPORTED

    def step(conv, cs=A16, w=A16):
        return L.ssm_conv_state_update(d, conv, cs, w, None, A16, A16, A16, A16, A16, A16, None,
                                       None, None, A16, None)

    assert step(L.make_conv_desc(4), cs=None) == L.SSM_ERR_INVALID_ARG      # width 4 needs a state
    assert step(L.make_conv_desc(4), w=None) == L.SSM_ERR_INVALID_ARG
    assert step(L.ssm_conv_desc(4, -1)) == L.SSM_ERR_INVALID_ARG
    assert step(L.make_conv_desc(4), cs=A16 + 2) == L.SSM_ERR_INVALID_ARG   # misaligned state


def test_options_rejections_before_launch(ssm_lib):
    L = ssm_lib
    d = L.make_desc(1, 8, 16, 16, L.SSM_DTYPE_F32)
    args = (A16, A16, A16, A16, A16, None, None, None, A16 + 4096, None, None, None, 0, None)
    assert L.ssm_scan_fwd_ex(d, None, *args) == L.SSM_ERR_INVALID_ARG           # no options
    assert L.ssm_scan_fwd_ex(d, L.make_opts(2), *args) == L.SSM_ERR_INVALID_ARG  # unknown
    o = L.make_opts("zoh")
    o.reserved[1] = 7
    assert L.ssm_scan_fwd_ex(d, o, *args) == L.SSM_ERR_INVALID_ARG             # reserved set
    assert L.ssm_scan_fwd_ex(L.make_desc(1, 8, 16, 3, 0), L.make_opts("zoh"), *args) \
        == L.SSM_ERR_UNSUPPORTED
    assert L.ssm_state_update_ex(d, L.make_opts(5), A16, A16, A16, A16, A16, A16, None, None,
                                 None, A16) == L.SSM_ERR_INVALID_ARG


def test_lti_rejections_before_launch(ssm_lib):
    L = ssm_lib
    d = L.make_desc(2, 64, 16, 16, L.SSM_DTYPE_F32)
    assert L.ssm_lti_kernel(L.make_desc(1, 64, 16, 3, 0), None, A16, A16, A16, A16, A16) \
        == L.SSM_ERR_UNSUPPORTED
    assert L.ssm_lti_kernel(d, L.make_opts(9), A16, A16, A16, A16, A16) == L.SSM_ERR_INVALID_ARG
    assert L.ssm_lti_kernel(d, None, A16 + 2, A16, A16, A16, A16) == L.SSM_ERR_INVALID_ARG
    assert L.ssm_lti_kernel(d, None, None, A16, A16, A16, A16) == L.SSM_ERR_INVALID_ARG
    assert L.ssm_lti_conv_fwd(d, A16, A16 + 2, None, None, A16) == L.SSM_ERR_INVALID_ARG
    assert L.ssm_lti_conv_fwd(d, None, A16, None, None, A16) == L.SSM_ERR_INVALID_ARG
    assert L.ssm_lti_conv_fwd(L.make_desc(0, 64, 16, 1, 0), A16, A16, None, None, A16) == L.SSM_OK


def test_bwd_plan_query(ssm_lib):
    """ssm_scan_bwd_plan: warps per CTA chosen so the CTAs spread evenly over
    the 148 SMs (one wave), its workspace equals the size query's, and it
    rejects what the size query rejects.  dstate 16 with 16-byte rows takes
    the one-warp-layout sweep (16 channels a warp, up to 7 warps a CTA in
    bf16 and 6 in fp32); other dstates the sweep of 32 / (dstate / 4) channels a warp."""
    bf = torch.bfloat16
    big = ssm_lib.make_desc(4, 8192, 4096, 16, bf)         # Mamba-1.4B layer
    pl = ssm_lib.ssm_scan_bwd_plan(big)
    assert (pl.nchunk, pl.warps, pl.channels, pl.ctas) == (1, 7, 112, 148)
    pl = ssm_lib.ssm_scan_bwd_plan(ssm_lib.make_desc(8, 2048, 1536, 16, bf))   # Mamba-130M layer
    assert (pl.nchunk, pl.warps, pl.channels, pl.ctas) == (1, 6, 96, 128)
    pl = ssm_lib.ssm_scan_bwd_plan(ssm_lib.make_desc(1, 262144, 2048, 16, bf))  # few channels, long
    assert pl.nchunk > 1 and pl.ctas * pl.warps <= 148 * 8    # every warp in one wave
    pl = ssm_lib.ssm_scan_bwd_plan(ssm_lib.make_desc(4, 8192, 4096, 64, bf))
    assert pl.channels == 2 * pl.warps                 # 16 lanes a channel at dstate 64
    for d in (big, ssm_lib.make_desc(2, 300, 72, 16, torch.float32),
              ssm_lib.make_desc(4, 8192, 4096, 16, torch.float32),
              ssm_lib.make_desc(4, 8192, 4096, 64, bf), ssm_lib.make_desc(1, 40, 5000, 8, bf)):
        for ck in (False, True):
            pl = ssm_lib.ssm_scan_bwd_plan(d, ck)
            assert pl.workspace == ssm_lib.ssm_scan_bwd_ex_workspace_size(d, ck)
            assert pl.ctas == pl.nchunk * d.batch * -(-d.dim // pl.channels)
            if d.dstate == 16:
                assert pl.channels == 16 * pl.warps
                assert pl.warps <= (7 if d.io_dtype == ssm_lib.SSM_DTYPE_BF16 else 6)
            else:
                assert pl.ctas <= 148 * (65536 // (pl.warps * 32 * 128)) or pl.warps == 8
    empty = ssm_lib.ssm_scan_bwd_plan(ssm_lib.make_desc(0, 10, 16, 16, bf))
    assert empty.ctas == 0 and empty.workspace == 0
    bad = ssm_lib.make_desc(1, 10, 16, 3, bf)
    info = ssm_lib.ssm_scan_bwd_plan_info()
    assert ssm_lib.lib.ssm_scan_bwd_plan(ctypes.byref(bad), 0, ctypes.byref(info)) == ssm_lib.SSM_ERR_UNSUPPORTED
    assert ssm_lib.lib.ssm_scan_bwd_plan(ctypes.byref(big), 0, None) == ssm_lib.SSM_ERR_INVALID_ARG
