"""The allocation-free look-back entry point against the context-based one.

sn_scan_lookback_noalloc serves callers that cannot allocate device memory at
run time (a fixed memory budget, an allocator that owns the device, a host
that forbids cudaMalloc after start-up).  It keeps its scratch in a
file-scope device array that every call shares.  This file runs last so a
failure here leaves every other test already run; it must pass both on its
own in a fresh process and after the rest of the suite (the shared array then
holds an earlier call's contents).
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


def _nrel(x, r):
    x, r = np.asarray(x, np.float64), np.asarray(r, np.float64)
    return float(np.max(np.abs(x - r)) / max(float(np.max(np.abs(r))), 1e-30))


def _with_ctx(sr, gated, a, rhs, s0):
    B, T, N = a.shape
    ctx = sr.Context(0)
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    ctx.ensure_workspace(B, T, N)
    fn = ctx.scan_gated if gated else ctx.scan_fma
    so, sf = fn(a, rhs, s0)
    torch.cuda.synchronize()
    assert ctx.last_error() == sr.SN_OK
    ctx.close()
    return so.cpu().numpy(), sf.cpu().numpy()


def _noalloc(sr, gated, a, rhs, s0):
    B, T, N = a.shape
    so = torch.full((B, T, N), float("nan"), device="cuda")
    sf = torch.full((B, N), float("nan"), device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    st = sr.sn_scan_lookback_noalloc(gated, B, T, N, a, rhs, s0, sf, so, status)
    assert st == sr.SN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == sr.SN_OK
    return so.cpu().numpy(), sf.cpu().numpy()


def test_no_alloc_matches_workspace_entry_point_on_two_calls(sr):
    # two calls in a row with different shapes and forms: the second one
    # finds the first one's flags and carries in the shared array
    for (B, T, N, gated, cid) in ((2, 3000, 96, 0, 201), (3, 1100, 64, 1, 202)):
        x = synth.scan_inputs(B, T, N, large=True, cid=cid)
        a, rhs = x["a"].cuda(), (x["u"] if gated else x["b"]).cuda()
        s0 = synth.normal((B, N), cid + 7).cuda()
        so_ref, sf_ref = _with_ctx(sr, gated, a, rhs, s0)
        so, sf = _noalloc(sr, gated, a, rhs, s0)
        # the same kernel and fold order as the context's look-back path: the same bits
        assert np.array_equal(so, so_ref) and np.array_equal(sf, sf_ref)
        # and the definition within the scans' tolerance
        ref = oracle.scan_gated if gated else oracle.scan_fma
        r64, f64 = ref(x["a"].numpy(), (x["u"] if gated else x["b"]).numpy(), s0.cpu().numpy().astype(np.float64))
        assert _nrel(so, r64) <= TOL and _nrel(sf, f64) <= TOL


def test_no_alloc_after_a_shape_change_and_back(sr):
    """Calls alternating between two tile counts: each change of tile count
    clears the flag and carry areas, and every call still gives the bits of
    the context's look-back path."""
    shapes = ((1, 2048, 64, 301), (2, 1024, 32, 302))
    ins = []
    for (B, T, N, cid) in shapes:
        x = synth.scan_inputs(B, T, N, large=True, cid=cid)
        ins.append((x["a"].cuda(), x["b"].cuda(), synth.normal((B, N), cid + 7).cuda()))
    refs = [_with_ctx(sr, 0, a, b, s0) for a, b, s0 in ins]
    for i in (0, 1, 0, 1):
        so, sf = _noalloc(sr, 0, *ins[i])
        assert np.array_equal(so, refs[i][0]) and np.array_equal(sf, refs[i][1])


def test_no_alloc_rejects_problems_beyond_its_scratch(sr):
    a = torch.zeros(4, device="cuda")
    T = 128 * (sr.SN_NOALLOC_MAX_TILES + 1)          # one channel block, one tile too many
    assert sr.sn_scan_lookback_noalloc(0, 1, T, 32, a, a, None, None, None) == sr.SN_E_NOMEM
    assert sr.sn_scan_lookback_noalloc(0, 1, 16, 30, a, a, None, None, None) == sr.SN_E_UNSUPPORTED
    assert sr.sn_scan_lookback_noalloc(2, 1, 16, 32, a, a, None, None, None) == sr.SN_E_INVAL


def test_no_alloc_replayed_from_a_cuda_graph(sr):
    """The allocation-free entry point captured in a CUDA graph (after a first,
    uncaptured call has set the device up) and replayed on new inputs: each
    replay equals an uncaptured call, because the launch epoch advances on
    the device."""
    B, T, N = 1, 8192, 64
    ins = []
    for i in range(3):
        x = synth.scan_inputs(B, T, N, large=True, cid=90 + i)
        ins.append((x["a"].cuda(), x["b"].cuda(), synth.normal((B, N), 9900 + i).cuda()))
    expect = [_noalloc(sr, 0, a, b, s0) for a, b, s0 in ins]
    a_d = torch.empty((B, T, N), device="cuda")
    b_d = torch.empty_like(a_d)
    s0_d = torch.empty((B, N), device="cuda")
    so = torch.empty_like(a_d)
    sf = torch.empty_like(s0_d)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert sr.sn_scan_lookback_noalloc(0, B, T, N, a_d, b_d, s0_d, sf, so, status) == sr.SN_OK
    for _ in range(2):
        for (a, b, s0), (eo, ef) in zip(ins, expect):
            a_d.copy_(a)
            b_d.copy_(b)
            s0_d.copy_(s0)
            g.replay()
            torch.cuda.synchronize()
            assert int(status.item()) == sr.SN_OK
            assert np.array_equal(so.cpu().numpy(), eo) and np.array_equal(sf.cpu().numpy(), ef)
