"""GPU parity of the reverse (adjoint) scans against the CPU oracle.

Both forms of "SunnyNet 工程化实录" §2.1, backward pass (the kernels' reverse
scan, §8).  The kernel uses the fp32 oracle's operation order, so it must
match it bit for bit, and stay within 1e-5 normwise of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def sr():
    import scan_runtime_gb300 as sr
    sr.build()
    return sr


@pytest.fixture()
def ctx(sr):
    c = sr.Context(0)
    yield c
    assert c.last_error() == sr.SN_OK
    c.close()


def _nrel(x, r):
    x, r = np.asarray(x, np.float64), np.asarray(r, np.float64)
    return float(np.max(np.abs(x - r)) / max(float(np.max(np.abs(r))), 1e-30))


def _case(B, T, N, seed, with_s0=True, with_gf=True):
    x = synth.scan_inputs(B, T, N, large=True, cid=300 + seed)
    s0 = synth.normal((B, N), 9300 + seed) if with_s0 else None
    gs = synth.normal((B, T, N), 9400 + seed)
    gf = synth.normal((B, N), 9500 + seed) if with_gf else None
    return x, s0, gs, gf


def _run(ctx, form, x, s, s0, gs, gf):
    rhs = x["u"] if form == "gated" else None
    cu = lambda t: None if t is None else t.cuda()
    ga, gb, g0 = ctx.scan_backward(form, cu(x["a"]), cu(s), cu(gs), s0=cu(s0), grad_final=cu(gf), u=cu(rhs))
    torch.cuda.synchronize()
    return ga.cpu().numpy(), gb.cpu().numpy(), g0.cpu().numpy()


def _forward32(form, x, s0):
    f = oracle.scan_fma if form == "fma" else oracle.scan_gated
    rhs = x["b"] if form == "fma" else x["u"]
    s, _ = f(x["a"].numpy(), rhs.numpy(), None if s0 is None else s0.numpy(), prec="f32")
    return torch.from_numpy(s)


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(2, 128, 128), (3, 77, 100), (1, 1, 64), (2, 33, 8), (1, 300, 4),
                                   (2, 65, 130), (1, 31, 7)])
@pytest.mark.parametrize("opts", [(True, True), (False, False)])
def test_backward_bit_exact_and_within_tolerance(ctx, form, shape, opts):
    B, T, N = shape
    x, s0, gs, gf = _case(B, T, N, sum(shape) % 61, *opts)
    s = _forward32(form, x, s0)
    ga, gb, g0 = _run(ctx, form, x, s, s0, gs, gf)
    u = x["u"].numpy() if form == "gated" else None
    args = (form, x["a"].numpy(), s.numpy())
    r32 = oracle.scan_backward(*args, None if s0 is None else s0.numpy(), gs.numpy(),
                               None if gf is None else gf.numpy(), u=u, prec="f32")
    r64 = oracle.scan_backward(form, x["a"].numpy(), s.numpy().astype(np.float64),
                               None if s0 is None else s0.numpy().astype(np.float64), gs.numpy(),
                               None if gf is None else gf.numpy(), u=u)
    for got, e32, e64 in zip((ga, gb, g0), r32, r64):
        assert np.array_equal(got.view(np.uint32), e32.view(np.uint32))
        assert _nrel(got, e64) <= TOL


def test_backward_optional_outputs(sr, ctx):
    B, T, N = 2, 40, 64
    x, s0, gs, gf = _case(B, T, N, 7)
    s = _forward32("fma", x, s0).cuda()
    gb = torch.full((B, T, N), 9.0, device="cuda")
    st = sr.sn_scan_fma_backward(ctx.handle, B, T, N, x["a"].cuda(), s0.cuda(), s, gs.cuda(), gf.cuda(),
                                 None, gb, None)
    assert st == sr.SN_OK
    torch.cuda.synchronize()
    _, e32, _ = oracle.scan_backward("fma", x["a"].numpy(), s.cpu().numpy(), s0.numpy(), gs.numpy(),
                                     gf.numpy(), prec="f32")
    assert np.array_equal(gb.cpu().numpy(), e32)


def test_backward_invalid_arguments(sr, ctx):
    a = torch.zeros(1, 8, 4, device="cuda")
    out = torch.full_like(a, 2.0)
    E = sr.SN_E_INVAL
    assert sr.sn_scan_fma_backward(ctx.handle, 1, 8, 4, a, None, None, a, None, out, None, None) == E  # no s
    assert sr.sn_scan_gated_backward(ctx.handle, 1, 8, 4, a, None, None, a, a, None, out, None, None) == E  # no u
    assert sr.sn_scan_fma_backward(ctx.handle, 1, 8, 4, a, None, a, a, None, a, None, None) == E  # out = in
    torch.cuda.synchronize()
    assert bool((out == 2.0).all())


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_full_size_backward_sampled(ctx, form):
    """B=8 T=8192 N=2048 in the benchmark's launch configuration; sampled
    channels recomputed by the oracle."""
    x = synth.config_inputs("scan_large")
    B, T, N = x["a"].shape
    gs = synth.normal((B, T, N), 9600)
    gf = synth.normal((B, N), 9601)
    fn = ctx.scan_fma if form == "fma" else ctx.scan_gated
    rhs = x["b"] if form == "fma" else x["u"]
    s, _ = fn(x["a"].cuda(), rhs.cuda(), x["s0"].cuda())
    ga, gb, g0 = ctx.scan_backward(form, x["a"].cuda(), s, gs.cuda(), s0=x["s0"].cuda(), grad_final=gf.cuda(),
                                   u=x["u"].cuda() if form == "gated" else None)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    for _ in range(10):
        bi, n = int(rng.integers(B)), int(rng.integers(N))
        col = lambda t: np.ascontiguousarray(t[bi, :, n].cpu().numpy()[None, :, None])
        r32 = oracle.scan_backward(form, col(x["a"]), col(s), x["s0"][bi, n].numpy().reshape(1, 1),
                                   col(gs), gf[bi, n].numpy().reshape(1, 1),
                                   u=col(x["u"]) if form == "gated" else None, prec="f32")
        assert np.array_equal(ga[bi, :, n].cpu().numpy(), r32[0][0, :, 0])
        assert np.array_equal(gb[bi, :, n].cpu().numpy(), r32[1][0, :, 0])
        assert g0[bi, n].item() == r32[2][0, 0]


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(1, 4096, 32), (2, 1000, 64), (1, 40000, 36), (3, 257, 96), (2, 5, 8)])
@pytest.mark.parametrize("opts", [(True, True), (False, False)])
def test_chunked_backward_within_tolerance(sr, ctx, form, shape, opts):
    """The chunked reverse scan (few channels, long T): per-tile reverse
    aggregates, a carry chain from the last chunk down, then the gradients.
    Its rounding order differs from the sequential kernel's, so it is held to
    the fp64 definition's tolerance, and two runs must agree bit for bit.
    T = 40000 spans several blocks of the carry chain and a ragged last chunk;
    T = 5 a single partial chunk."""
    B, T, N = shape
    x, s0, gs, gf = _case(B, T, N, 17 + T % 13, *opts)
    s = _forward32(form, x, s0)
    ctx.ensure_workspace(B, T, N)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
    first = _run(ctx, form, x, s, s0, gs, gf)
    second = _run(ctx, form, x, s, s0, gs, gf)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    u = x["u"].numpy() if form == "gated" else None
    r64 = oracle.scan_backward(form, x["a"].numpy(), s.numpy().astype(np.float64),
                               None if s0 is None else s0.numpy().astype(np.float64), gs.numpy(),
                               None if gf is None else gf.numpy(), u=u)
    for got, again, e64 in zip(first, second, r64):
        assert np.array_equal(got, again)
        assert _nrel(got, e64) <= TOL


def test_chunked_backward_optional_outputs_and_auto(sr, ctx):
    """grad_a, grad_b and grad_s0 may each be NULL; with a workspace set and few
    channels the automatic choice takes the chunked path (same bits as forcing it)."""
    B, T, N = 1, 3000, 32
    x, s0, gs, gf = _case(B, T, N, 23)
    s = _forward32("fma", x, s0)
    ctx.ensure_workspace(B, T, N)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
    ga, gb, g0 = _run(ctx, "fma", x, s, s0, gs, gf)
    a, sd, gsd, s0d, gfd = (t.cuda() for t in (x["a"], s, gs, s0, gf))
    only_b = torch.full((B, T, N), 7.0, device="cuda")
    assert sr.sn_scan_fma_backward(ctx.handle, B, T, N, a, s0d, sd, gsd, gfd, None, only_b, None) == sr.SN_OK
    torch.cuda.synchronize()
    assert np.array_equal(only_b.cpu().numpy(), gb)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    ga2, gb2, g02 = _run(ctx, "fma", x, s, s0, gs, gf)
    assert np.array_equal(ga2, ga) and np.array_equal(gb2, gb) and np.array_equal(g02, g0)


def test_auto_keeps_sequential_for_many_channels(sr, ctx):
    """Eight batches of 2048 channels give the sequential reverse scan enough
    CTAs: with a workspace set, the automatic choice still takes it (its bits,
    which differ from the chunked path's)."""
    B, T, N = 8, 1024, 2048
    x, s0, gs, gf = _case(B, T, N, 29)
    s = _forward32("fma", x, s0)
    ctx.ensure_workspace(B, T, N)
    outs = {}
    for k in (sr.SN_SCAN_KERNEL_AUTO, sr.SN_SCAN_KERNEL_SEQUENTIAL, sr.SN_SCAN_KERNEL_REDUCE_SCAN):
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, k)
        outs[k] = _run(ctx, "fma", x, s, s0, gs, gf)[0]
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    assert not np.array_equal(outs[sr.SN_SCAN_KERNEL_SEQUENTIAL], outs[sr.SN_SCAN_KERNEL_REDUCE_SCAN])
    assert np.array_equal(outs[sr.SN_SCAN_KERNEL_AUTO], outs[sr.SN_SCAN_KERNEL_SEQUENTIAL])
