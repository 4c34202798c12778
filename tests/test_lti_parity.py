"""GPU parity of the time-invariant model's convolution mode: ssm_lti_kernel
(the kernel K) and ssm_lti_conv_fwd (y = K * x + D x, gated) against the fp64
oracle, through the C ABI.  Bounds: K (fp32 output) and y with fp32 I/O
elementwise 1e-4 (1 + |ref|); y with bf16 I/O 1e-2 (1 + |ref|)."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, f64, rel_err
from selective_state_space_137_b300 import ops, synth

pytestmark = pytest.mark.gpu


def lti_params(dim, N, seed):
    r = np.random.default_rng(seed)
    delta = r.uniform(1e-3, 0.3, dim).astype(np.float32)
    A = (-np.exp(np.log(np.arange(1, N + 1))[None, :].repeat(dim, 0)
                 + r.uniform(-0.3, 0.3, (dim, N)))).astype(np.float32)
    B = r.standard_normal((dim, N)).astype(np.float32)
    C = r.standard_normal((dim, N)).astype(np.float32)
    return delta, A, B, C


@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("N", [1, 4, 16, 64])
def test_lti_kernel(cuda, disc, N):
    dim, L = 40, 300
    delta, A, B, C = lti_params(dim, N, 10 + N)
    K = ops.lti_kernel(*(torch.from_numpy(a).to(cuda) for a in (delta, A, B, C)), L,
                       discretization=disc)
    torch.cuda.synchronize()
    ref = oracle.lti_kernel(delta, A, B, C, L, zoh=disc == "zoh")
    assert rel_err(f64(K), ref) <= 1e-4


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 300, 72), (1, 1, 8), (3, 63, 40), (1, 129, 33)])
def test_lti_conv(cuda, io, shape):
    bsz, L, dim = shape
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[io]
    delta, A, B, C = lti_params(dim, 16, 5 + L)
    Kref = oracle.lti_kernel(delta, A, B, C, L)
    g = torch.Generator().manual_seed(L + dim)
    x = torch.randn((bsz, L, dim), generator=g).to(dt)
    z = torch.randn((bsz, L, dim), generator=g).to(dt)
    D = torch.randn(dim, generator=g)
    K32 = torch.from_numpy(Kref.astype(np.float32))
    y = ops.lti_conv_fwd(K32.to(cuda), x.to(cuda), D=D.to(cuda), z=z.to(cuda))
    y0 = ops.lti_conv_fwd(K32.to(cuda), x.to(cuda))
    torch.cuda.synchronize()
    ref = oracle.lti_conv(f64(K32), f64(x), D=f64(D), z=f64(z))
    ref0 = oracle.lti_conv(f64(K32), f64(x))
    assert rel_err(f64(y), ref) <= TOL[dt]
    assert rel_err(f64(y0), ref0) <= TOL[dt]


def test_lti_conv_many_items_per_cta(cuda):
    """bf16 with 16-byte rows takes the tensor-core kernel, whose persistent
    CTAs each take several (channel block, step group) items of different
    weights: 2 sequences (a partial block of 8), 900 steps (8 groups of 128,
    the last partial), 1024 channels, with D and the gate."""
    bsz, L, dim = 2, 900, 1024
    delta, A, B, C = lti_params(dim, 16, 91)
    K32 = torch.from_numpy(oracle.lti_kernel(delta, A, B, C, L).astype(np.float32))
    g = torch.Generator().manual_seed(19)
    x = torch.randn((bsz, L, dim), generator=g).to(torch.bfloat16)
    z = torch.randn((bsz, L, dim), generator=g).to(torch.bfloat16)
    D = torch.randn(dim, generator=g)
    y = ops.lti_conv_fwd(K32.to(cuda), x.to(cuda), D=D.to(cuda), z=z.to(cuda))
    torch.cuda.synchronize()
    ref = oracle.lti_conv(f64(K32), f64(x), D=f64(D), z=f64(z))
    assert rel_err(f64(y), ref) <= TOL[torch.bfloat16]


def test_lti_conv_mode_equals_recurrence(cuda):
    """Convolution mode (kernel + conv) and the recurrence (ssm_scan_fwd with
    the constant step, B and C shared by all channels) give the same output."""
    bsz, L, dim, N = 2, 500, 64, 16
    delta, A, B, C = lti_params(dim, N, 77)
    B[:] = B[0]
    C[:] = C[0]
    t = lambda a: torch.from_numpy(a).to(cuda)
    g = torch.Generator().manual_seed(3)
    x = torch.randn((bsz, L, dim), generator=g).to(cuda)
    K = ops.lti_kernel(t(delta), t(A), t(B), t(C), L)
    y_conv = ops.lti_conv_fwd(K, x)
    dl = t(delta)[None, None, :].expand(bsz, L, dim).contiguous()
    Bs = t(B[0])[None, None, :].expand(bsz, L, N).contiguous()
    Cs = t(C[0])[None, None, :].expand(bsz, L, N).contiguous()
    y_rec, _ = ops.scan_fwd(x, dl, t(A), Bs, Cs, delta_softplus=False)
    torch.cuda.synchronize()
    assert rel_err(f64(y_conv), f64(y_rec)) <= 1e-4


def test_lti_full_size_sampled(cuda):
    """The Mamba-130M layer (8 x 2048 x 1536, N = 16) in convolution mode with
    the inputs the benchmark draws: the kernel K of sampled channels against
    the oracle's closed form, and y = K * x on those channels against the
    oracle's convolution with the same fp32 K."""
    from parity import sample_channels
    w = synth.MAMBA_130M
    g = torch.Generator(device=cuda).manual_seed(5)
    N = w.dstate
    delta = 0.001 + 0.1 * torch.rand(w.dim, generator=g, device=cuda)
    A = -torch.arange(1, N + 1, device=cuda, dtype=torch.float32).repeat(w.dim, 1).contiguous()
    Bv = torch.randn(N, generator=g, device=cuda)
    Cv = torch.randn(N, generator=g, device=cuda)
    Bp, Cp = Bv.repeat(w.dim, 1).contiguous(), Cv.repeat(w.dim, 1).contiguous()
    x = torch.randn((w.batch, w.seqlen, w.dim), generator=g, device=cuda).to(torch.bfloat16)
    K = ops.lti_kernel(delta, A, Bp, Cp, w.seqlen)
    y = ops.lti_conv_fwd(K, x)
    torch.cuda.synchronize()
    for b, ds in sample_channels(w.batch, w.dim):
        idx = torch.tensor(ds, device=cuda)
        sel = lambda t: f64(t.index_select(0, idx))
        Kref = oracle.lti_kernel(sel(delta), sel(A), sel(Bp), sel(Cp), w.seqlen)
        assert rel_err(sel(K), Kref) <= 1e-4, (b, ds)
        ref = oracle.lti_conv(sel(K), f64(x[b:b + 1].index_select(-1, idx)))
        assert rel_err(f64(y[b:b + 1].index_select(-1, idx)), ref) <= TOL[torch.bfloat16], (b, ds)


def test_lti_conv_full_size_slow_decay_sampled(cuda):
    """The longest convolution-mode workload (8 x 2048 x 1536, bf16) with the
    slowest decay (Delta in [1e-3, 2e-3], so K stays near its first tap over
    all 2048 steps), D and the gate: where a single bf16 term per tap drifts
    furthest, the tensor-core kernel's hi + lo terms must hold the bf16
    bound.  Sampled channels of sampled sequences against the oracle run on
    those channels alone."""
    from parity import sample_channels
    bsz, L, dim = 8, 2048, 1536
    delta, A, B, C = lti_params(dim, 16, 123)
    delta[:] = np.random.default_rng(124).uniform(1e-3, 2e-3, dim).astype(np.float32)
    g = torch.Generator(device=cuda).manual_seed(125)
    x = torch.randn((bsz, L, dim), generator=g, device=cuda).to(torch.bfloat16)
    z = torch.randn((bsz, L, dim), generator=g, device=cuda).to(torch.bfloat16)
    D = torch.randn(dim, generator=g, device=cuda)
    t = lambda a: torch.from_numpy(a).to(cuda)
    K = ops.lti_kernel(t(delta), t(A), t(B), t(C), L)
    y = ops.lti_conv_fwd(K, x, D=D, z=z)
    torch.cuda.synchronize()
    for b, ds in sample_channels(bsz, dim):
        idx = torch.tensor(ds, device=cuda)
        pick = lambda a: f64(a[b:b + 1].index_select(-1, idx))
        ref = oracle.lti_conv(f64(K.index_select(0, idx)), pick(x), D=f64(D.index_select(0, idx)), z=pick(z))
        assert rel_err(pick(y), ref) <= TOL[torch.bfloat16], (b, ds)
