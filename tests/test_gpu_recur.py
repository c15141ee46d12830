"""GPU parity of the tier-2 matrix recurrences (through the C ABI).

Bar: o and the final state within 1e-4 normwise of the fp64 oracle; the
diagonal-decay state bit-exact with the single-precision definition (its
update has no reduction); bit-exact segment splits within the GPU path
("SunnyNet 工程化实录" §4); hand fixtures reproduced exactly; per-head value
slices independent with dk != dv (the bug of the llama.cpp comparison
article §3); grouped k/q for the Mamba-2 shape (§4.1).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _golden

pytestmark = pytest.mark.gpu

TOL = 1e-4


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


def cu(t):
    return None if t is None else t.cuda()


def _np(t):
    return t.cpu().numpy() if t is not None else None


def _f64(t):
    return None if t is None else t.numpy().astype(np.float64)


# ------------------------------------------------------------------ per-kind runners
def run_diag(ctx, x, S0=None, **kw):
    o, S = ctx.recur_diag(*(cu(x[n]) for n in ("q", "k", "v", "d")), cu(S0), H=x["H"], G=x["G"],
                          decay_kind=x["decay_kind"], scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return _np(o), _np(S)


def ref_diag(x, S0=None, prec="f64"):
    S0 = (_f64(S0) if prec == "f64" else (None if S0 is None else S0.numpy()))
    return oracle.recur_diag(*(x[n].numpy() for n in ("q", "k", "v", "d")), S0, H=x["H"], G=x["G"],
                             decay_kind=x["decay_kind"], scale=x["scale"], prec=prec)


def run_delta(ctx, x, S0=None, **kw):
    o, S = ctx.recur_delta(*(cu(x[n]) for n in ("q", "k", "v", "beta")), cu(S0), scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return _np(o), _np(S)


def ref_delta(x, S0=None):
    return oracle.recur_delta(*(x[n].numpy() for n in ("q", "k", "v", "beta")), _f64(S0), scale=x["scale"])


def run_rwkv(ctx, x, S0=None, **kw):
    o, S = ctx.recur_rwkv7(*(cu(x[n]) for n in ("q", "k", "v", "w")), cu(S0), **kw)
    torch.cuda.synchronize()
    return _np(o), _np(S)


def ref_rwkv(x, S0=None):
    return oracle.recur_rwkv7(*(x[n].numpy() for n in ("q", "k", "v", "w")), _f64(S0))


def make(kind, B, T, H, dk, dv, G=None, seed=0):
    if kind in ("gated_key", "gated_head"):
        return synth.gated_memory_inputs(B, T, H, dk, dv, per_key=(kind == "gated_key"), cid=100 + seed)
    if kind == "gla":
        return synth.gla_inputs(B, T, H, dk, dv, cid=60 + seed)
    if kind == "mamba2":
        return synth.mamba2_inputs(B, T, H, G or 1, dk, dv, cid=70 + seed)
    if kind == "delta":
        return synth.deltanet_inputs(B, T, H, dk, dv, cid=80 + seed)
    return synth.rwkv7_inputs(B, T, H, dk, dv, cid=90 + seed)


RUN = {"gla": (run_diag, ref_diag), "mamba2": (run_diag, ref_diag), "delta": (run_delta, ref_delta),
       "rwkv": (run_rwkv, ref_rwkv), "gated_key": (run_diag, ref_diag), "gated_head": (run_diag, ref_diag)}


def state_shape(kind, B, H, dk, dv):
    return (B, H, dv, dk) if kind == "rwkv" else (B, H, dk, dv)


# ------------------------------------------------------------------ parity
@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv", "gated_key", "gated_head"])
@pytest.mark.parametrize("dims", [(128, 128), (128, 64), (64, 128), (64, 64)])
@pytest.mark.parametrize("T", [1, 2, 37, 100])
def test_parity_small(ctx, kind, dims, T):
    dk, dv = dims
    B, H = 2, 4
    x = make(kind, B, T, H, dk, dv, G=2 if kind == "mamba2" else None, seed=T % 7)
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5000 + T) * 0.5
    run, ref = RUN[kind]
    o, S = run(ctx, x, S0)
    ro, rS = ref(x, S0)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2", "gated_key", "gated_head"])
def test_diag_state_is_bit_exact_with_single_precision_definition(ctx, kind):
    x = make(kind, 2, 50, 4, 128, 64, G=1, seed=3)
    S0 = synth.normal((2, 4, 128, 64), 5100)
    _, S = run_diag(ctx, x, S0)
    _, rS = ref_diag(x, S0, prec="f32")
    assert np.array_equal(S.view(np.uint32), rS.view(np.uint32))


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv"])
def test_optional_outputs_and_in_place_state(ctx, kind):
    B, T, H, dk, dv = 1, 20, 2, 64, 128
    x = make(kind, B, T, H, dk, dv, seed=4)
    run, ref = RUN[kind]
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5200)
    ro, rS = ref(x, S0)
    o, S = run(ctx, x, S0, o=None)
    assert o is None and _nrel(S, rS) <= TOL
    o, S = run(ctx, x, S0, S_out=None)
    assert S is None and _nrel(o, ro) <= TOL
    st = S0.cuda()
    kw = dict(S_out=st)
    if kind in ("gla", "mamba2"):
        ctx.recur_diag(*(cu(x[n]) for n in ("q", "k", "v", "d")), st, H=x["H"], G=x["G"],
                       decay_kind=x["decay_kind"], scale=x["scale"], **kw)
    elif kind == "delta":
        ctx.recur_delta(*(cu(x[n]) for n in ("q", "k", "v", "beta")), st, scale=x["scale"], **kw)
    else:
        ctx.recur_rwkv7(*(cu(x[n]) for n in ("q", "k", "v", "w")), st, **kw)
    torch.cuda.synchronize()
    assert _nrel(st.cpu().numpy(), rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv", "gated_key"])
@pytest.mark.parametrize("split", [1, 19, 48])
def test_segment_split_bit_exact(ctx, kind, split):
    B, T, H, dk, dv = 2, 64, 2, 128 if kind != "rwkv" else 64, 64
    x = make(kind, B, T, H, dk, dv, seed=5)
    run, _ = RUN[kind]
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5300)
    of, Sf = run(ctx, x, S0)
    tk = ("q", "k", "v", "d") if kind in ("gla", "mamba2", "gated_key") else ("q", "k", "v", "beta") \
        if kind == "delta" else ("q", "k", "v", "w")
    x1 = dict(x, **{n: x[n][:, :split].contiguous() for n in tk})
    x2 = dict(x, **{n: x[n][:, split:].contiguous() for n in tk})
    o1, S1 = run(ctx, x1, S0)
    o2, S2 = run(ctx, x2, torch.from_numpy(S1))
    assert np.array_equal(np.concatenate([o1, o2], 1), of) and np.array_equal(S2, Sf)


@pytest.mark.parametrize("kind", ["gla", "delta", "rwkv"])
def test_head_value_slices_independent(ctx, kind):
    """dk != dv; perturbing head 1's v changes head 1 only (bitwise)."""
    B, T, H, dk, dv = 1, 24, 3, 128 if kind != "rwkv" else 64, 64 if kind != "rwkv" else 128
    x = make(kind, B, T, H, dk, dv, seed=6)
    run, _ = RUN[kind]
    o1, S1 = run(ctx, x)
    x2 = dict(x)
    x2["v"] = x["v"].clone()
    x2["v"][:, :, 1] += 1.0
    o2, S2 = run(ctx, x2)
    for h in (0, 2):
        assert np.array_equal(o1[:, :, h], o2[:, :, h]) and np.array_equal(S1[:, h], S2[:, h])
    assert not np.allclose(o1[:, :, 1], o2[:, :, 1])


def test_grouped_keys_equal_replicated(ctx):
    x = make("mamba2", 2, 30, 6, 128, 64, G=2, seed=7)
    o1, S1 = run_diag(ctx, x)
    rep = torch.tensor([0, 0, 0, 1, 1, 1])
    x2 = dict(x, q=x["q"][:, :, rep].contiguous(), k=x["k"][:, :, rep].contiguous(), G=6)
    o2, S2 = run_diag(ctx, x2)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


# ------------------------------------------------------------------ hand fixtures
def _embed(vals, shape, big_shape):
    out = np.zeros(big_shape, np.float32)
    out[tuple(slice(0, s) for s in shape)] = np.asarray(vals, np.float32).reshape(shape)
    return torch.from_numpy(out)


def test_hand_fixtures_exact(ctx):
    """The dyadic hand-derived examples, zero-padded into 64 x 64 heads, come
    back exactly (every intermediate value is exactly representable)."""
    D = 64
    g = _golden.load("diag_gla_dyadic.txt")
    B, T, H, G, dk, dv = g["shape"]
    x = dict(q=_embed(g["q"], (B, T, G, dk), (B, T, G, D)), k=_embed(g["k"], (B, T, G, dk), (B, T, G, D)),
             v=_embed(g["v"], (B, T, H, dv), (B, T, H, D)), H=H, G=G, decay_kind=0, scale=1.0)
    d = np.ones((B, T, H, D), np.float32)
    d[..., :dk] = np.asarray(g["d"], np.float32).reshape(B, T, H, dk)
    x["d"] = torch.from_numpy(d)
    o, S = run_diag(ctx, x)
    assert np.array_equal(o[..., :dv].ravel(), np.asarray(g["o"], np.float32))
    assert np.array_equal(S[:, :, :dk, :dv].ravel(), np.asarray(g["S"], np.float32))

    g = _golden.load("diag_mamba2_dyadic.txt")
    B, T, H, G, dk, dv = g["shape"]
    x = dict(q=_embed(g["q"], (B, T, G, dk), (B, T, G, D)), k=_embed(g["k"], (B, T, G, dk), (B, T, G, D)),
             v=_embed(g["v"], (B, T, H, dv), (B, T, H, D)), d=_embed(g["d"], (B, T, H), (B, T, H)),
             H=H, G=G, decay_kind=1, scale=1.0)
    o, S = run_diag(ctx, x)
    assert np.array_equal(o[..., :dv].ravel(), np.asarray(g["o"], np.float32))
    assert np.array_equal(S[:, :, :dk, :dv].ravel(), np.asarray(g["S"], np.float32))

    g = _golden.load("diag_gated_dyadic.txt")
    B, T, H, G, dk, dv = g["shape"]
    x = dict(q=_embed(g["q"], (B, T, G, dk), (B, T, G, D)), k=_embed(g["k"], (B, T, G, dk), (B, T, G, D)),
             v=_embed(g["v"], (B, T, H, dv), (B, T, H, D)), H=H, G=G, decay_kind=2, scale=1.0)
    d = np.ones((B, T, H, D), np.float32)
    d[..., :dk] = np.asarray(g["d"], np.float32).reshape(B, T, H, dk)
    x["d"] = torch.from_numpy(d)
    o, S = run_diag(ctx, x, _embed(g["S0"], (B, H, dk, dv), (B, H, D, D)))
    assert np.array_equal(o[..., :dv].ravel(), np.asarray(g["o"], np.float32))
    assert np.array_equal(S[:, :, :dk, :dv].ravel(), np.asarray(g["S"], np.float32))

    g = _golden.load("delta_dyadic.txt")
    B, T, H, dk, dv = g["shape"]
    x = dict(q=_embed(g["q"], (B, T, H, dk), (B, T, H, D)), k=_embed(g["k"], (B, T, H, dk), (B, T, H, D)),
             v=_embed(g["v"], (B, T, H, dv), (B, T, H, D)), beta=_embed(g["beta"], (B, T, H), (B, T, H)),
             scale=1.0)
    o, S = run_delta(ctx, x, _embed(g["S0"], (B, H, dk, dv), (B, H, D, D)))
    assert np.array_equal(o[..., :dv].ravel(), np.asarray(g["o"], np.float32))
    assert np.array_equal(S[:, :, :dk, :dv].ravel(), np.asarray(g["S"], np.float32))

    g = _golden.load("rwkv7_dyadic.txt")
    B, T, H, dk, dv = g["shape"]
    w = np.ones((B, T, H, D), np.float32)
    w[..., :dk] = np.asarray(g["w"], np.float32).reshape(B, T, H, dk)
    x = dict(q=_embed(g["q"], (B, T, H, dk), (B, T, H, D)), k=_embed(g["k"], (B, T, H, dk), (B, T, H, D)),
             v=_embed(g["v"], (B, T, H, dv), (B, T, H, D)), w=torch.from_numpy(w))
    o, S = run_rwkv(ctx, x, _embed(g["S0"], (B, H, dv, dk), (B, H, D, D)))
    assert np.array_equal(o[..., :dv].ravel(), np.asarray(g["o"], np.float32))
    assert np.array_equal(S[:, :, :dv, :dk].ravel(), np.asarray(g["S"], np.float32))


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("B", [1, 3, 37])
def test_rwkv7_decode_parity_and_in_place(ctx, B):
    H = 12
    x = synth.rwkv7_inputs(B, 1, H, 64, 64, random_state=True, cid=95)
    o, S = run_rwkv(ctx, x, x["S0"])
    ro, rS = ref_rwkv(x, x["S0"])
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL
    st = x["S0"].cuda()
    o2, _ = ctx.recur_rwkv7(*(cu(x[n]) for n in ("q", "k", "v", "w")), st, S_out=st)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), S) and np.array_equal(o2.cpu().numpy(), o)
    o3, S3 = run_rwkv(ctx, x, None)
    ro3, rS3 = ref_rwkv(x, None)
    assert _nrel(o3, ro3) <= TOL and _nrel(S3, rS3) <= TOL


def test_decode_matches_sequence_kernel_at_t1(sr, ctx):
    x = synth.rwkv7_inputs(8, 1, 12, 64, 64, random_state=True, cid=96)
    o1, S1 = run_rwkv(ctx, x, x["S0"])
    ctx.set_option(sr.SN_OPT_RECUR_KERNEL, 1)
    o2, S2 = run_rwkv(ctx, x, x["S0"])
    ro, rS = ref_rwkv(x, x["S0"])
    assert _nrel(o1, ro) <= TOL and _nrel(o2, ro) <= TOL and _nrel(S2, rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "gated_key", "gated_head", "rwkv"])
@pytest.mark.parametrize("dims", [(128, 128), (128, 64), (64, 64), (64, 128)])
def test_column_decode_matches_sequence_kernel_bit_for_bit(sr, ctx, kind, dims):
    """T = 1 of every kind runs the column decode kernel, which sums in the
    sequence kernel's order for the same call (rows per lane); a forced
    one-step sequence call must give the same bits for o and the state."""
    dk, dv = dims
    B, H = 64, 4
    x = make(kind, B, 1, H, dk, dv, G=2 if kind == "mamba2" else None, seed=11)
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5300) * 0.5
    run, ref = RUN[kind]
    o1, S1 = run(ctx, x, S0)
    ctx.set_option(sr.SN_OPT_RECUR_KERNEL, 1)
    o2, S2 = run(ctx, x, S0)
    ctx.set_option(sr.SN_OPT_RECUR_KERNEL, 0)
    assert np.array_equal(S1, S2) and np.array_equal(o1, o2)
    ro, rS = ref(x, S0)
    assert _nrel(o1, ro) <= TOL and _nrel(S1, rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "delta", "gated_head"])
def test_column_decode_in_place_and_optional_outputs(ctx, kind):
    B, H, dk, dv = 5, 3, 128, 128
    x = make(kind, B, 1, H, dk, dv, seed=12)
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5400) * 0.5
    run, ref = RUN[kind]
    o, S = run(ctx, x, S0)
    st = S0.cuda()
    names = ("q", "k", "v", "d") if kind != "delta" else ("q", "k", "v", "beta")
    args = [cu(x[n]) for n in names]
    if kind == "delta":
        o2, _ = ctx.recur_delta(*args, st, scale=x["scale"], S_out=st)
    else:
        o2, _ = ctx.recur_diag(*args, st, H=x["H"], G=x["G"], decay_kind=x["decay_kind"], scale=x["scale"], S_out=st)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), S) and np.array_equal(o2.cpu().numpy(), o)
    o3, S3 = run(ctx, x, S0, o=False)
    assert o3 is None and np.array_equal(S3, S)
    o4, S4 = run(ctx, x, None)
    ro4, rS4 = ref(x, None)
    assert _nrel(o4, ro4) <= TOL and _nrel(S4, rS4) <= TOL


# ------------------------------------------------------------------ validation
def test_invalid_arguments(sr, ctx):
    h = ctx.handle
    q = torch.zeros(1, 4, 2, 64, device="cuda")
    v = torch.zeros(1, 4, 2, 64, device="cuda")
    g = torch.zeros(1, 4, 2, device="cuda")
    o = torch.full((1, 4, 2, 64), 5.0, device="cuda")
    assert sr.sn_recur_diag(h, 1, 4, 2, 2, 32, 64, 0, 1.0, q, q, v, q, None, None, o) == sr.SN_E_UNSUPPORTED
    assert sr.sn_recur_diag(h, 1, 4, 3, 2, 64, 64, 1, 1.0, q, q, v, g, None, None, o) == sr.SN_E_INVAL
    assert sr.sn_recur_diag(h, 1, 4, 2, 2, 64, 64, 7, 1.0, q, q, v, q, None, None, o) == sr.SN_E_INVAL
    assert sr.sn_recur_delta(h, 1, 4, 2, 64, 64, 1.0, q, q, v, g, None, None, q) == sr.SN_E_INVAL
    assert sr.sn_recur_delta(h, 1, 0, 2, 64, 64, 1.0, q, q, v, g, None, None, o) == sr.SN_E_INVAL
    assert sr.sn_recur_rwkv7(h, 1, 4, 2, 64, 64, q.data_ptr() + 4, q, v, q, None, None, o) == sr.SN_E_INVAL
    assert sr.sn_recur_rwkv7(h, 1, 4, 2, 64, 96, q, q, v, q, None, None, o) == sr.SN_E_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 5.0).all())


# ------------------------------------------------------------------ full-size workloads
def _sample_heads(B, H, n, seed):
    rng = np.random.default_rng(seed)
    return sorted({(int(rng.integers(B)), int(rng.integers(H))) for _ in range(n)} | {(0, 0), (B - 1, H - 1)})


@pytest.mark.parametrize("name", ["gla", "mamba2", "deltanet", "rwkv7_prefill"])
def test_full_size_sampled_heads(ctx, name):
    """Full-size workloads in the launch configuration the benchmark times;
    sampled (b, h) sequences recomputed one by one by the oracle."""
    x = synth.config_inputs(name)
    c = synth.CONFIGS[name]
    B, H = c["B"], c["H"]
    if name in ("gla", "mamba2"):
        o, S = run_diag(ctx, x)
    elif name == "deltanet":
        o, S = run_delta(ctx, x)
    else:
        o, S = run_rwkv(ctx, x)
    for (b, h) in _sample_heads(B, H, 3, 21):
        if name in ("gla", "mamba2"):
            G = x["G"]
            g = h // (H // G)
            xs = dict(x, q=x["q"][b:b + 1, :, g:g + 1].contiguous(), k=x["k"][b:b + 1, :, g:g + 1].contiguous(),
                      v=x["v"][b:b + 1, :, h:h + 1].contiguous(), H=1, G=1,
                      d=(x["d"][b:b + 1, :, h:h + 1].contiguous()))
            ro, rS = ref_diag(xs)
        elif name == "deltanet":
            xs = {n: x[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "beta")}
            xs["scale"] = x["scale"]
            ro, rS = ref_delta(xs)
        else:
            xs = {n: x[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "w")}
            ro, rS = ref_rwkv(xs)
        assert _nrel(o[b:b + 1, :, h:h + 1], ro) <= TOL
        assert _nrel(S[b:b + 1, h:h + 1], rS) <= TOL


def test_full_size_rwkv7_decode(ctx):
    x = synth.config_inputs("rwkv7_decode")
    o, S = run_rwkv(ctx, x, x["S0"])
    idx = np.random.default_rng(22).choice(1024, 16, replace=False)
    xs = {n: x[n][idx].contiguous() for n in ("q", "k", "v", "w", "S0")}
    ro, rS = ref_rwkv(xs, xs["S0"])
    assert _nrel(o[idx], ro) <= TOL and _nrel(S[idx], rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv"])
def test_cta_widths_give_identical_bits(sr, ctx, kind):
    """The CTA width only tiles the value columns; every width returns the
    same bits, and matches the oracle."""
    B, T, H = 2, 40, 2
    dk = 64 if kind == "rwkv" else 128
    dv = 128
    x = make(kind, B, T, H, dk, dv, G=1 if kind == "mamba2" else None, seed=8)
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5400)
    run, ref = RUN[kind]
    outs = []
    for w in (0, 2, 4, 8):
        ctx.set_option(sr.SN_OPT_RECUR_TILE, w)
        outs.append(run(ctx, x, S0))
    ctx.set_option(sr.SN_OPT_RECUR_TILE, 0)
    for o, S in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(S, outs[0][1])
    ro, rS = ref(x, S0)
    assert _nrel(outs[0][0], ro) <= TOL and _nrel(outs[0][1], rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2", "delta", "rwkv"])
def test_forced_widths_on_64_value_columns(sr, ctx, kind):
    """Every CTA width (2, 4, 8 warps) tiles a 64-column value dimension, is
    accepted on the host and gives the automatic width's bits."""
    B, T, H, dv = 2, 37, 2, 64
    dk = 64 if kind == "rwkv" else 128
    x = make(kind, B, T, H, dk, dv, G=1 if kind == "mamba2" else None, seed=9)
    S0 = synth.normal(state_shape(kind, B, H, dk, dv), 5401)
    run, ref = RUN[kind]
    outs = []
    try:
        for w in (0, 2, 4, 8):
            ctx.set_option(sr.SN_OPT_RECUR_TILE, w)
            outs.append(run(ctx, x, S0))
    finally:
        ctx.set_option(sr.SN_OPT_RECUR_TILE, 0)
    for o, S in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(S, outs[0][1])
    ro, rS = ref(x, S0)
    assert _nrel(outs[0][0], ro) <= TOL and _nrel(outs[0][1], rS) <= TOL
