"""GPU parity of the readout epilogues (sn_readout_norm_gate, sn_readout_dskip)
against the fp64 oracle: within 1e-5 normwise, in place allowed, every row
count (ragged against the rows a warp handles), both head sizes, and the
full GLA and Mamba-2 output shapes."""
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
    r = np.asarray(r, np.float64)
    return float(np.max(np.abs(x - r)) / max(float(np.max(np.abs(r))), 1e-30))


@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 37, 3), (3, 101, 4)])
@pytest.mark.parametrize("with_w", [True, False])
def test_norm_gate_parity(ctx, dv, shape, with_w):
    B, T, H = shape
    o = synth.normal((B, T, H, dv), 900 + T) * 0.7
    g = synth.normal((B, T, H, dv), 901 + T, 0.0, 2.0)
    w = synth.normal((dv,), 902, 1.0, 0.3) if with_w else None
    y = ctx.readout_norm_gate(o.cuda(), g.cuda(), None if w is None else w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.readout_norm_gate(o.numpy(), g.numpy(), None if w is None else w.numpy(), eps=1e-6)
    assert _nrel(y.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("dv", [64, 128])
def test_norm_gate_in_place_and_extreme_gates(ctx, dv):
    B, T, H = 2, 50, 2
    o = synth.normal((B, T, H, dv), 910)
    g = synth.normal((B, T, H, dv), 911, 0.0, 30.0)       # silu saturates at both ends
    ref = oracle.readout_norm_gate(o.numpy(), g.numpy(), None, eps=1e-5)
    od = o.cuda()
    y = ctx.readout_norm_gate(od, g.cuda(), eps=1e-5, y=od)
    torch.cuda.synchronize()
    assert y.data_ptr() == od.data_ptr()
    assert _nrel(od.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 37, 3), (4, 300, 24)])
def test_dskip_parity_and_in_place(ctx, dv, shape):
    B, T, H = shape
    o = synth.normal((B, T, H, dv), 920 + T)
    x = synth.normal((B, T, H, dv), 921 + T)
    D = synth.normal((H,), 922)
    ref = oracle.readout_dskip(o.numpy(), x.numpy(), D.numpy())
    y = ctx.readout_dskip(o.cuda(), x.cuda(), D.cuda())
    od = o.cuda()
    ctx.readout_dskip(od, x.cuda(), D.cuda(), y=od)
    torch.cuda.synchronize()
    assert _nrel(y.cpu().numpy(), ref) <= TOL
    assert np.array_equal(od.cpu().numpy(), y.cpu().numpy())


def test_full_size_outputs(ctx):
    """The GLA (B4 T4096 H4 dv128) and Mamba-2 (B4 T4096 H24 dv64) output shapes."""
    o = synth.normal((4, 4096, 4, 128), 930)
    g = synth.normal((4, 4096, 4, 128), 931)
    w = synth.normal((128,), 932, 1.0, 0.2)
    y = ctx.readout_norm_gate(o.cuda(), g.cuda(), w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    assert _nrel(y.cpu().numpy(), oracle.readout_norm_gate(o.numpy(), g.numpy(), w.numpy(), eps=1e-6)) <= TOL
    o = synth.normal((4, 4096, 24, 64), 933)
    x = synth.normal((4, 4096, 24, 64), 934)
    D = synth.normal((24,), 935)
    y = ctx.readout_dskip(o.cuda(), x.cuda(), D.cuda())
    torch.cuda.synchronize()
    assert _nrel(y.cpu().numpy(), oracle.readout_dskip(o.numpy(), x.numpy(), D.numpy())) <= TOL


def test_invalid_arguments(ctx, sr):
    abi = sr._abi
    o = torch.zeros((1, 2, 1, 64), device="cuda")
    g = torch.zeros((1, 2, 1, 64), device="cuda")
    assert abi.sn_readout_norm_gate(ctx.handle, 1, 2, 1, 64, o, g, None, -1.0, o) == sr.SN_E_INVAL
    assert abi.sn_readout_norm_gate(ctx.handle, 1, 2, 1, 64, o, g, None, float("nan"), o) == sr.SN_E_INVAL
    assert abi.sn_readout_norm_gate(ctx.handle, 1, 2, 1, 32, o, g, None, 1e-6, o) == sr.SN_E_UNSUPPORTED
    assert abi.sn_readout_norm_gate(ctx.handle, 1, 2, 1, 64, o, g, None, 1e-6, g) == sr.SN_E_INVAL   # y overlaps g
    assert abi.sn_readout_dskip(ctx.handle, 1, 2, 1, 64, o, g, None, o) == sr.SN_E_INVAL
    torch.cuda.synchronize()
