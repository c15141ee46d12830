"""GPU parity of the tier-1 scans (through the C ABI) against the CPU oracle.

Bar ("SunnyNet 工程化实录" §2.1 forms, §4 segment continuation):
* the sequential kernel equals the single-precision definition bit for bit
  (fp32 oracle with one fused multiply-add per step) and is split-invariant;
* every kernel is within 1e-5 normwise of the fp64 oracle;
* the look-back kernel is deterministic and bit-exact under splits at
  multiples of its chunk length.
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
    x = np.asarray(x, np.float64)
    return float(np.max(np.abs(x - r)) / max(float(np.max(np.abs(r))), 1e-30))


def _inputs(B, T, N, seed, large=True):
    x = synth.scan_inputs(B, T, N, large=large, cid=50 + seed)
    s0 = synth.normal((B, N), 9000 + seed)
    return x["a"], x["b"], x["u"], s0


def _run(ctx, form, a, rhs, s0, **kw):
    fn = ctx.scan_fma if form == "fma" else ctx.scan_gated
    so, sf = fn(a.cuda(), rhs.cuda(), None if s0 is None else s0.cuda(), **kw)
    torch.cuda.synchronize()
    return (None if so is None else so.cpu().numpy()), (None if sf is None else sf.cpu().numpy())


def _ref(form, a, rhs, s0, prec):
    fn = oracle.scan_fma if form == "fma" else oracle.scan_gated
    if s0 is not None:
        s0 = s0.numpy() if prec == "f32" else s0.numpy().astype(np.float64)
    return fn(a.numpy(), rhs.numpy(), s0, prec=prec)


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(2, 128, 128), (3, 77, 100), (1, 1, 64), (2, 2, 8), (1, 300, 4),
                                   (2, 65, 130), (1, 33, 7), (4, 40, 1)])
def test_sequential_bit_exact_and_within_tolerance(ctx, form, shape):
    B, T, N = shape
    a, b, u, s0 = _inputs(B, T, N, hash(shape) % 97)
    rhs = b if form == "fma" else u
    so, sf = _run(ctx, form, a, rhs, s0)
    r32, f32 = _ref(form, a, rhs, s0, "f32")
    r64, f64 = _ref(form, a, rhs, s0, "f64")
    assert np.array_equal(so.view(np.uint32), r32.view(np.uint32))
    assert np.array_equal(sf.view(np.uint32), f32.view(np.uint32))
    assert _nrel(so, r64) <= TOL and _nrel(sf, f64) <= TOL


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(1024, 1, 2048), (1, 1, 2048), (3, 1, 7), (5, 1, 130)])
def test_single_step_bit_exact_in_place_and_views(ctx, form, shape):
    """T = 1 (the single-step entry) runs its own elementwise kernel with the
    sequential kernel's arithmetic: the fp32 definition's bits, in place
    (s_final == s0), without s0, and on unaligned views (plain-load path)."""
    B, T, N = shape
    a, b, u, s0 = _inputs(B, T, N, 40 + N % 11)
    rhs = b if form == "fma" else u
    so, sf = _run(ctx, form, a, rhs, s0)
    r32, f32 = _ref(form, a, rhs, s0, "f32")
    assert np.array_equal(so, r32) and np.array_equal(sf, f32)
    fn = ctx.scan_fma if form == "fma" else ctx.scan_gated
    st = s0.cuda().clone()
    fn(a.cuda(), rhs.cuda(), st, s_out=None, s_final=st)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), f32)
    so0, _ = _run(ctx, form, a, rhs, None)
    assert np.array_equal(so0, _ref(form, a, rhs, None, "f32")[0])
    big_a, big_r = torch.zeros(B * N + 1), torch.zeros(B * N + 1)
    big_a[1:] = a.reshape(-1)
    big_r[1:] = rhs.reshape(-1)
    so1, sf1 = fn(big_a.cuda()[1:].view(B, T, N), big_r.cuda()[1:].view(B, T, N), s0.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(so1.cpu().numpy(), r32) and np.array_equal(sf1.cpu().numpy(), f32)


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_small_workload_config(ctx, form):
    """B=2 T=128 N=128, a = sigmoid(N(0,1)), s0 = 0 (the pages' parity size)."""
    x = synth.config_inputs("scan_small")
    rhs = x["b"] if form == "fma" else x["u"]
    so, sf = _run(ctx, form, x["a"], rhs, None)
    r32, _ = _ref(form, x["a"], rhs, None, "f32")
    r64, f64 = _ref(form, x["a"], rhs, None, "f64")
    assert np.array_equal(so, r32)
    assert _nrel(so, r64) <= TOL and _nrel(sf, f64) <= TOL


def test_unaligned_views_take_the_plain_load_path(ctx):
    B, T, N = 2, 50, 64
    a, b, _, s0 = _inputs(B, T, N, 3)
    big_a = torch.zeros(B * T * N + 1)
    big_b = torch.zeros(B * T * N + 1)
    big_a[1:] = a.reshape(-1)
    big_b[1:] = b.reshape(-1)
    ga, gb = big_a.cuda()[1:].view(B, T, N), big_b.cuda()[1:].view(B, T, N)
    so, sf = ctx.scan_fma(ga, gb, s0.cuda())
    r32, f32 = _ref("fma", a, b, s0, "f32")
    assert np.array_equal(so.cpu().numpy(), r32) and np.array_equal(sf.cpu().numpy(), f32)


def test_optional_outputs_and_in_place_state(ctx):
    B, T, N = 2, 70, 64
    a, b, _, s0 = _inputs(B, T, N, 4)
    _, f32 = _ref("fma", a, b, s0, "f32")
    so, sf = _run(ctx, "fma", a, b, s0, s_out=None)
    assert so is None and np.array_equal(sf, f32)
    st = s0.cuda().clone()
    ctx.scan_fma(a.cuda(), b.cuda(), st, s_out=None, s_final=st)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), f32)
    so, sf = _run(ctx, "fma", a, b, s0, s_final=None)
    assert sf is None


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("split", [1, 77, 150])
def test_sequential_segment_split_bit_exact(ctx, form, split):
    B, T, N = 2, 300, 192
    a, b, u, s0 = _inputs(B, T, N, 5)
    rhs = b if form == "fma" else u
    full, ffull = _run(ctx, form, a, rhs, s0)
    p1, f1 = _run(ctx, form, a[:, :split].contiguous(), rhs[:, :split].contiguous(), s0)
    p2, f2 = _run(ctx, form, a[:, split:].contiguous(), rhs[:, split:].contiguous(), torch.from_numpy(f1))
    assert np.array_equal(np.concatenate([p1, p2], 1), full) and np.array_equal(f2, ffull)


# ------------------------------------------------------------------ look-back kernel
@pytest.fixture()
def lbctx(sr, ctx):
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    return ctx


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(1, 4096, 32), (2, 1000, 64), (3, 257, 96), (1, 256, 32), (2, 5, 8),
                                   (1, 70000, 64)])
def test_lookback_within_tolerance(lbctx, form, shape):
    B, T, N = shape
    lbctx.ensure_workspace(B, T, N)
    a, b, u, s0 = _inputs(B, T, N, 6 + T % 13)
    rhs = b if form == "fma" else u
    so, sf = _run(lbctx, form, a, rhs, s0)
    r64, f64 = _ref(form, a, rhs, s0, "f64")
    assert _nrel(so, r64) <= TOL and _nrel(sf, f64) <= TOL
    assert np.array_equal(so[:, -1], sf)


def test_lookback_deterministic(lbctx):
    B, T, N = 1, 20000, 64
    lbctx.ensure_workspace(B, T, N)
    a, b, _, s0 = _inputs(B, T, N, 7)
    r1 = _run(lbctx, "fma", a, b, s0)
    r2 = _run(lbctx, "fma", a, b, s0)
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])


def _replay_matches(sr, call, ins, expect):
    """Capture `call` (on fixed device buffers) in a CUDA graph, then replay it
    on each input set twice over: the outputs must equal `expect` bit for bit."""
    B, T, N = ins[0][0].shape
    a_d = torch.empty((B, T, N), device="cuda")
    b_d = torch.empty_like(a_d)
    s0_d = torch.empty((B, N), device="cuda")
    so = torch.empty_like(a_d)
    sf = torch.empty_like(s0_d)
    a_d.copy_(ins[0][0])
    b_d.copy_(ins[0][1])
    s0_d.copy_(ins[0][2])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert call(a_d, b_d, s0_d, sf, so) == sr.SN_OK
    for _ in range(2):
        for (a, b, s0), (eo, ef) in zip(ins, expect):
            a_d.copy_(a)
            b_d.copy_(b)
            s0_d.copy_(s0)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(so.cpu().numpy(), eo) and np.array_equal(sf.cpu().numpy(), ef)


def test_lookback_replayed_from_a_cuda_graph(sr, lbctx):
    """A captured look-back call replayed on new inputs: every replay must
    publish its chunk flags under a fresh tag (the launch epoch is kept and
    advanced on the device), else a replay would take the previous replay's
    carries as published.  Each replay equals an uncaptured call."""
    B, T, N = 1, 8192, 64
    lbctx.ensure_workspace(B, T, N)
    ins = [(a, b, s0) for a, b, _, s0 in (_inputs(B, T, N, 30 + i) for i in range(3))]
    expect = [_run(lbctx, "fma", a, b, s0) for a, b, s0 in ins]
    call = lambda a, b, s0, sf, so: sr.sn_scan_fma(lbctx.handle, B, T, N, a, b, s0, sf, so)
    _replay_matches(sr, call, ins, expect)
    assert lbctx.last_error() == sr.SN_OK


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_lookback_split_at_chunk_multiple_bit_exact(sr, lbctx, form):
    tc = lbctx.get_option(sr.SN_OPT_LOOKBACK_CHUNK)
    B, T, N = 2, 20 * tc + 17, 64
    split = 12 * tc
    lbctx.ensure_workspace(B, T, N)
    a, b, u, s0 = _inputs(B, T, N, 8)
    rhs = b if form == "fma" else u
    full, ffull = _run(lbctx, form, a, rhs, s0)
    p1, f1 = _run(lbctx, form, a[:, :split].contiguous(), rhs[:, :split].contiguous(), s0)
    p2, f2 = _run(lbctx, form, a[:, split:].contiguous(), rhs[:, split:].contiguous(), torch.from_numpy(f1))
    assert np.array_equal(np.concatenate([p1, p2], 1), full) and np.array_equal(f2, ffull)


def test_lookback_bounded_wait_reports_timeout(sr, lbctx):
    """A flag that no chunk publishes: every wait runs out after the limit, the
    kernel returns normally and the context reports SN_E_TIMEOUT once."""
    B, T, N = 1, 4 * 128, 32
    lbctx.ensure_workspace(B, T, N)
    lbctx.set_option(sr.SN_OPT_WAIT_LIMIT_US, 2000)
    lbctx.set_option(sr.SN_OPT_DEBUG_POISON, 1)
    a, b, _, s0 = _inputs(B, T, N, 9)
    _run(lbctx, "fma", a, b, s0)
    assert lbctx.last_error() == sr.SN_E_TIMEOUT
    assert lbctx.last_error() == sr.SN_OK             # cleared
    lbctx.set_option(sr.SN_OPT_DEBUG_POISON, 0)
    so, sf = _run(lbctx, "fma", a, b, s0)              # context still usable
    r64, f64 = _ref("fma", a, b, s0, "f64")
    assert _nrel(so, r64) <= TOL


@pytest.mark.parametrize("form", ["fma", "gated"])
@pytest.mark.parametrize("shape", [(1, 4096, 32), (2, 1000, 64), (3, 257, 96), (2, 5, 8), (1, 70000, 64),
                                   (1, 40000, 36), (1, 70000, 32), (4, 4096, 1024), (2, 16384, 512)])
def test_reduce_scan_matches_lookback_bit_for_bit(sr, ctx, form, shape):
    """The reduce-then-scan path and the fused path run the look-back kernel's
    local scans, aggregates and carry chain in the same order, so their
    results equal the look-back's bit for bit; T = 70000 and 40000 span
    several blocks of the carry chains and wrap their rings, N = 36 is a
    ragged channel tile, (1, 70000, 32) a single column, and the last two
    have so many columns that the fused path's aggregates run far ahead."""
    B, T, N = shape
    ctx.ensure_workspace(B, T, N)
    a, b, u, s0 = _inputs(B, T, N, 40 + T % 11)
    rhs = b if form == "fma" else u
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    lo, lf = _run(ctx, form, a, rhs, s0)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
    ro, rf = _run(ctx, form, a, rhs, s0)
    ro0, rf0 = _run(ctx, form, a, rhs, None)
    ctx.ensure_workspace_bytes(sr.sn_workspace_bytes(sr.SN_OP_SCAN_FMA, B, T, N) + 4096)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_FUSED)
    fo, ff = _run(ctx, form, a, rhs, s0)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    assert np.array_equal(ro, lo) and np.array_equal(rf, lf)
    assert np.array_equal(fo, lo) and np.array_equal(ff, lf)
    r64, f64 = _ref(form, a, rhs, s0, "f64")
    assert _nrel(ro, r64) <= TOL and _nrel(rf, f64) <= TOL
    z64, zf64 = _ref(form, a, rhs, None, "f64")
    assert _nrel(ro0, z64) <= TOL and _nrel(rf0, zf64) <= TOL


def test_fused_random_shapes_repeated_bit_equal(sr, ctx):
    """Seeded shapes across the fused path's regimes (one to several columns,
    ragged T and N, with and without s0, both forms), each run three times in
    a row: every run gives the reduce-then-scan bits (the carries are read
    through tagged words with no fence, so a race would show as a
    difference)."""
    rng = np.random.default_rng(2024)
    for case in range(10):
        B = int(rng.integers(1, 4))
        N = int(rng.integers(1, 41)) * 4
        T = int(rng.integers(1024, 90000))
        form = "fma" if case % 2 == 0 else "gated"
        ctx.ensure_workspace(B, T, N)
        a, b, u, s0 = _inputs(B, T, N, 500 + case)
        rhs = b if form == "fma" else u
        s0 = s0 if case % 3 else None
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
        ro, rf = _run(ctx, form, a, rhs, s0)
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_FUSED)
        for _ in range(3):
            fo, ff = _run(ctx, form, a, rhs, s0)
            assert np.array_equal(fo, ro) and np.array_equal(ff, rf), (B, T, N, form)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)


def test_fused_bounded_wait_reports_timeout(sr, lbctx):
    """The fused kernel's state tiles wait for a carry state no CTA writes:
    the first wait runs out after the limit, the others stop at the abort,
    the kernel returns and the context reports SN_E_TIMEOUT once; the next
    call works."""
    B, T, N = 1, 40000, 64
    lbctx.ensure_workspace(B, T, N)
    lbctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_FUSED)
    lbctx.set_option(sr.SN_OPT_WAIT_LIMIT_US, 2000)
    lbctx.set_option(sr.SN_OPT_DEBUG_POISON, 1)
    a, b, _, s0 = _inputs(B, T, N, 10)
    _run(lbctx, "fma", a, b, s0)
    assert lbctx.last_error() == sr.SN_E_TIMEOUT
    assert lbctx.last_error() == sr.SN_OK             # cleared
    lbctx.set_option(sr.SN_OPT_DEBUG_POISON, 0)
    so, sf = _run(lbctx, "fma", a, b, s0)              # context still usable
    assert lbctx.last_error() == sr.SN_OK
    r64, f64 = _ref("fma", a, b, s0, "f64")
    assert _nrel(so, r64) <= TOL and _nrel(sf, f64) <= TOL


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_fused_optional_outputs_match_reduce_scan(sr, ctx, form):
    """The fused path without s0 (zeros), and with the final state alone (no
    s_out), gives the reduce-then-scan path's bits."""
    B, T, N = 1, 40000, 64
    ctx.ensure_workspace(B, T, N)
    a, b, u, _ = _inputs(B, T, N, 43)
    rhs = b if form == "fma" else u
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
    ro, rf = _run(ctx, form, a, rhs, None)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_FUSED)
    fo, ff = _run(ctx, form, a, rhs, None)
    fnone, fonly = _run(ctx, form, a, rhs, None, s_out=False)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    assert ctx.last_error() == sr.SN_OK
    assert np.array_equal(fo, ro) and np.array_equal(ff, rf)
    assert fnone is None and np.array_equal(fonly, rf)


def test_reduce_scan_optional_outputs_and_split(sr, ctx):
    tc = ctx.get_option(sr.SN_OPT_LOOKBACK_CHUNK)
    B, T, N = 2, 300 * tc + 9, 64
    split = 140 * tc
    ctx.ensure_workspace(B, T, N)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_REDUCE_SCAN)
    a, b, _, s0 = _inputs(B, T, N, 41)
    full, ffull = _run(ctx, "fma", a, b, s0)
    none_out, f_only = _run(ctx, "fma", a, b, s0, s_out=False)
    p1, f1 = _run(ctx, "fma", a[:, :split].contiguous(), b[:, :split].contiguous(), s0)
    p2, f2 = _run(ctx, "fma", a[:, split:].contiguous(), b[:, split:].contiguous(), torch.from_numpy(f1))
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    assert none_out is None and np.array_equal(f_only, ffull)
    assert np.array_equal(np.concatenate([p1, p2], 1), full) and np.array_equal(f2, ffull)


def test_lookback_forced_without_workspace_is_nomem(sr, ctx):
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    a = torch.zeros(1, 512, 32, device="cuda")
    out = torch.full_like(a, 7.0)
    s = sr.sn_scan_fma(ctx.handle, 1, 512, 32, a, a, None, None, out)
    assert s == sr.SN_E_NOMEM
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())                     # untouched


@pytest.mark.parametrize("kernel", ["lookback", "reduce_scan", "fused"])
@pytest.mark.parametrize("shape", [(1, 70000, 64), (2, 1000, 64), (1, 256, 32)])
def test_chunked_in_place_continuation(sr, ctx, kernel, shape):
    """s_final may be s0's buffer.  The chunked kernels read s0 before any tile
    writes a final state (the first chunk only; the output pass reads the
    chain's copy), so in place gives the out-of-place bits."""
    B, T, N = shape
    ctx.ensure_workspace_bytes(sr.sn_workspace_bytes(sr.SN_OP_SCAN_FMA, B, T, N) + 4096)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, {"lookback": sr.SN_SCAN_KERNEL_LOOKBACK,
                                           "reduce_scan": sr.SN_SCAN_KERNEL_REDUCE_SCAN,
                                           "fused": sr.SN_SCAN_KERNEL_FUSED}[kernel])
    a, b, _, s0 = _inputs(B, T, N, 71 + T % 7)
    a, b, s0 = a.cuda(), b.cuda(), s0.cuda()
    so1, sf1 = torch.empty_like(a), torch.empty_like(s0)
    assert sr.sn_scan_fma(ctx.handle, B, T, N, a, b, s0, sf1, so1) == sr.SN_OK
    st = s0.clone()
    so2 = torch.empty_like(a)
    assert sr.sn_scan_fma(ctx.handle, B, T, N, a, b, st, st, so2) == sr.SN_OK
    torch.cuda.synchronize()
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    assert torch.equal(so1, so2) and torch.equal(sf1, st)


def test_fused_interleaved_with_other_chunked_calls_and_shapes(sr, ctx):
    """The fused path keeps tagged flags where the look-back kernel keeps its
    own: calls of both kernels, reduce-then-scan calls and changes of shape
    on one context all give the look-back's bits."""
    shapes = ((1, 20000, 64), (2, 3000, 32), (1, 20000, 64))
    ins = [_inputs(*sh, 60 + i) for i, sh in enumerate(shapes)]
    ctx.ensure_workspace_bytes(max(sr.sn_workspace_bytes(sr.SN_OP_SCAN_FMA, *sh) for sh in shapes) + 4096)
    ref = []
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    for (a, b, _, s0) in ins:
        ref.append(_run(ctx, "fma", a, b, s0))
    order = [(0, sr.SN_SCAN_KERNEL_FUSED), (1, sr.SN_SCAN_KERNEL_FUSED), (1, sr.SN_SCAN_KERNEL_LOOKBACK),
             (1, sr.SN_SCAN_KERNEL_FUSED), (2, sr.SN_SCAN_KERNEL_REDUCE_SCAN), (2, sr.SN_SCAN_KERNEL_FUSED),
             (0, sr.SN_SCAN_KERNEL_FUSED), (0, sr.SN_SCAN_KERNEL_FUSED)]
    for i, kern in order:
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, kern)
        a, b, _, s0 = ins[i]
        so, sf = _run(ctx, "fma", a, b, s0)
        assert np.array_equal(so, ref[i][0]) and np.array_equal(sf, ref[i][1]), (i, kern)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)


def test_fused_replayed_from_a_cuda_graph(sr, ctx):
    """A fused call captured in a CUDA graph and replayed on new inputs: the
    launch epoch advances on the device, so each replay equals an uncaptured
    call bit for bit."""
    B, T, N = 1, 16384, 64
    ctx.ensure_workspace_bytes(sr.sn_workspace_bytes(sr.SN_OP_SCAN_FMA, B, T, N) + 4096)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_FUSED)
    ins = [tuple(t.cuda() for t in _inputs(B, T, N, 80 + i)) for i in range(3)]
    expect = [_run(ctx, "fma", a.cpu(), b.cpu(), s0.cpu()) for a, b, _, s0 in ins]
    a_d, b_d = torch.empty((B, T, N), device="cuda"), torch.empty((B, T, N), device="cuda")
    s0_d, so, sf = torch.empty((B, N), device="cuda"), torch.empty((B, T, N), device="cuda"), torch.empty((B, N), device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert sr.sn_scan_fma(ctx.handle, B, T, N, a_d, b_d, s0_d, sf, so) == sr.SN_OK
    for _ in range(2):
        for (a, b, _, s0), (eo, ef) in zip(ins, expect):
            a_d.copy_(a)
            b_d.copy_(b)
            s0_d.copy_(s0)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(so.cpu().numpy(), eo) and np.array_equal(sf.cpu().numpy(), ef)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)


def test_auto_choice_by_channel_count(sr, ctx):
    """With a workspace set, the automatic choice chunks along T only when the
    channels leave most SMs idle: one channel tile takes reduce-then-scan, eight
    batches of 2048 channels stay on the sequential kernel.  The two kernels
    round differently, so the bits show which one ran."""
    auto, seq, rs = sr.SN_SCAN_KERNEL_AUTO, sr.SN_SCAN_KERNEL_SEQUENTIAL, sr.SN_SCAN_KERNEL_REDUCE_SCAN
    for (B, T, N), want in (((1, 4096, 32), rs), ((8, 1024, 2048), seq)):
        a, b, _, s0 = _inputs(B, T, N, 61)
        ctx.ensure_workspace(B, T, N)
        outs = {}
        for k in (auto, seq, rs):
            ctx.set_option(sr.SN_OPT_SCAN_KERNEL, k)
            outs[k] = _run(ctx, "fma", a, b, s0)[0]
        assert not np.array_equal(outs[seq], outs[rs])
        assert np.array_equal(outs[auto], outs[want])
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, auto)


# ------------------------------------------------------------------ validation
def test_invalid_arguments_leave_outputs_untouched(sr, ctx):
    h = ctx.handle
    a = torch.randn(2, 16, 64, device="cuda")
    out = torch.full_like(a, 3.0)
    fin = torch.full((2, 64), 3.0, device="cuda")
    E = sr.SN_E_INVAL
    assert sr.sn_scan_fma(h, 0, 16, 64, a, a, None, fin, out) == E
    assert sr.sn_scan_fma(h, 2, -1, 64, a, a, None, fin, out) == E
    assert sr.sn_scan_fma(h, 2, 16, 64, None, a, None, fin, out) == E
    assert sr.sn_scan_fma(h, 2, 16, 64, a, a, None, fin, a) == E            # output aliases input
    assert sr.sn_scan_fma(h, 2, 16, 64, a, a, None, out, out) == E          # two outputs overlap
    assert sr.sn_scan_fma(h, 2, 16, 64, a.data_ptr() + 2, a, None, fin, out) == E   # misaligned
    assert sr.sn_scan_gated(h, 1 << 20, 1 << 20, 1 << 20, a, a, None, fin, out) == E  # element-count bound
    torch.cuda.synchronize()
    assert bool((out == 3.0).all()) and bool((fin == 3.0).all())


def test_options(sr, ctx):
    assert ctx.get_option(sr.SN_OPT_LOOKBACK_CHUNK) == 128
    assert sr.sn_ctx_set_option(ctx.handle, sr.SN_OPT_LOOKBACK_CHUNK, 5) == sr.SN_E_INVAL
    assert sr.sn_ctx_set_option(ctx.handle, sr.SN_OPT_SCAN_KERNEL, 9) == sr.SN_E_INVAL
    assert sr.sn_ctx_set_option(ctx.handle, 12345, 0) == sr.SN_E_INVAL
    ctx.set_option(sr.SN_OPT_WAIT_LIMIT_US, 500000)
    assert ctx.get_option(sr.SN_OPT_WAIT_LIMIT_US) == 500000


# ------------------------------------------------------------------ full-size workload
@pytest.fixture(scope="module")
def large_inputs():
    return synth.config_inputs("scan_large")


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_full_size_sequential_sampled_and_split(ctx, large_inputs, form):
    """B=8 T=8192 N=2048 in the launch configuration the benchmark times;
    sampled channels against the oracle and the 3000 + 5192 split."""
    x = large_inputs
    rhs = x["b"] if form == "fma" else x["u"]
    B, T, N = x["a"].shape
    ga, gr, gs0 = x["a"].cuda(), rhs.cuda(), x["s0"].cuda()
    fn = ctx.scan_fma if form == "fma" else ctx.scan_gated
    so, sf = fn(ga, gr, gs0)
    rng = np.random.default_rng(11)
    chans = [(int(rng.integers(B)), int(rng.integers(N))) for _ in range(24)] + [(0, 0), (B - 1, N - 1)]
    so_s = {c: so[c[0], :, c[1]].cpu().numpy() for c in chans}
    sf_h = sf.cpu().numpy()
    for c in chans:
        ac = np.ascontiguousarray(x["a"][c[0], :, c[1]].numpy()[None, :, None])
        rc = np.ascontiguousarray(rhs[c[0], :, c[1]].numpy()[None, :, None])
        s = x["s0"][c[0], c[1]].numpy().reshape(1, 1)
        f = oracle.scan_fma if form == "fma" else oracle.scan_gated
        r32, f32 = f(ac, rc, s, prec="f32")
        r64, _ = f(ac, rc, s.astype(np.float64))
        assert np.array_equal(so_s[c], r32[0, :, 0]) and sf_h[c] == f32[0, 0]
        assert _nrel(so_s[c], r64[0, :, 0]) <= TOL
    # split 3000 + 5192, state carried, equals the full run bit for bit
    p1, f1 = fn(ga[:, :3000].contiguous(), gr[:, :3000].contiguous(), gs0)
    p2, f2 = fn(ga[:, 3000:].contiguous(), gr[:, 3000:].contiguous(), f1)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([p1, p2], 1), so) and torch.equal(f2, sf)


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_full_size_lookback_sampled_and_split(sr, ctx, large_inputs, form):
    x = large_inputs
    rhs = x["b"] if form == "fma" else x["u"]
    B, T, N = x["a"].shape
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    ctx.ensure_workspace(B, T, N)
    ga, gr, gs0 = x["a"].cuda(), rhs.cuda(), x["s0"].cuda()
    fn = ctx.scan_fma if form == "fma" else ctx.scan_gated
    so, sf = fn(ga, gr, gs0)
    rng = np.random.default_rng(12)
    for _ in range(12):
        bi, n = int(rng.integers(B)), int(rng.integers(N))
        ac = np.ascontiguousarray(x["a"][bi, :, n].numpy()[None, :, None])
        rc = np.ascontiguousarray(rhs[bi, :, n].numpy()[None, :, None])
        s = x["s0"][bi, n].numpy().reshape(1, 1).astype(np.float64)
        r64, f64 = (oracle.scan_fma if form == "fma" else oracle.scan_gated)(ac, rc, s)
        assert _nrel(so[bi, :, n].cpu().numpy(), r64[0, :, 0]) <= TOL
    split = 3072                                        # a multiple of the 128-step chunk length
    p1, f1 = fn(ga[:, :split].contiguous(), gr[:, :split].contiguous(), gs0)
    p2, f2 = fn(ga[:, split:].contiguous(), gr[:, split:].contiguous(), f1)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([p1, p2], 1), so) and torch.equal(f2, sf)


def test_scan_host_pipeline_matches_device_path(ctx):
    """Context.scan_host (host buffers streamed through the GPU in batch-row
    chunks on three streams) returns the device path's bits for both forms."""
    B, T, N = 5, 300, 192
    a, b, u, s0 = _inputs(B, T, N, 12)
    outs = ctx.scan_host(a.pin_memory(), b.pin_memory(), u.pin_memory(), s0.pin_memory(), rows_per_chunk=2)
    for form, rhs in (("fma", b), ("gated", u)):
        so, sf = _run(ctx, form, a, rhs, s0)
        assert np.array_equal(outs[form][0].numpy(), so) and np.array_equal(outs[form][1].numpy(), sf)
    only = ctx.scan_host(a, u=u, s0=None)
    r32, _ = _ref("gated", a, u, None, "f32")
    assert set(only) == {"gated"} and np.array_equal(only["gated"][0].numpy(), r32)


def test_scan_host_rejects_bad_arguments_before_any_transfer(sr, ctx):
    """sn_scan_host checks its arguments on the host: no form, a staging
    buffer smaller than the query or not 256-byte aligned, an output that
    overlaps an input."""
    B, T, N = 3, 64, 32
    a, b, u, s0 = _inputs(B, T, N, 13)
    so = torch.zeros((B, T, N))
    sf = torch.zeros((B, N))
    need = sr.sn_scan_host_staging_bytes(B, T, N, 1, 1)
    need2 = sr.sn_scan_host_staging_bytes(B, T, N, 1, 2)
    stg = torch.empty(max(need, need2) + 512, dtype=torch.uint8, device="cuda")
    h = ctx.handle
    assert sr.sn_scan_host(h, B, T, N, 1, a, None, None, s0, so, sf, None, None, stg, need) == sr.SN_E_INVAL
    assert sr.sn_scan_host(h, B, T, N, 1, a, b, None, s0, so, sf, None, None, stg, need - 1) == sr.SN_E_INVAL
    assert sr.sn_scan_host(h, B, T, N, 1, a, b, None, s0, so, sf, None, None, stg[16:], need) == sr.SN_E_INVAL
    assert sr.sn_scan_host(h, B, T, N, 1, a, b, None, s0, a, sf, None, None, stg, need) == sr.SN_E_INVAL
    assert torch.count_nonzero(so) == 0 and torch.count_nonzero(sf) == 0
    # and a valid call on the caller's stream, pageable buffers, ragged last chunk
    s = torch.cuda.Stream()
    assert sr.sn_scan_host(h, B, T, N, 2, a, b, None, s0, so, sf, None, None, stg, need2, s) == sr.SN_OK
    s.synchronize()
    ref_so, ref_sf = _run(ctx, "fma", a, b, s0)
    assert np.array_equal(so.numpy(), ref_so) and np.array_equal(sf.numpy(), ref_sf)
