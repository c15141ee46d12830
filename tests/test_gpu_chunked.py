"""GPU parity of the chunked tensor-core form of the diagonal-decay recurrence
(sn_recur_diag_chunked) against the fp64 oracle.

Bar: o and the final state within 2e-3 normwise of the fp64 oracle (the
operands of the tensor-core products are tf32); splits at multiples of the
128-token chunk are bit-exact within the GPU path (the chunk grid does not
move); per-key decays strong enough to leave the single-anchor range are
evaluated exactly; non-positive decays are reported as SN_E_RANGE, never as
silently wrong numbers.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
CHUNK = 128


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


def make(kind, B, T, H, dv, G=None, seed=0):
    if kind == "gla":
        return synth.gla_inputs(B, T, H, 128, dv, cid=300 + seed)
    return synth.mamba2_inputs(B, T, H, G or 1, 128, dv, cid=310 + seed)


def run_chunked(ctx, x, S0=None, **kw):
    o, S = ctx.recur_diag_chunked(*(cu(x[n]) for n in ("q", "k", "v", "d")), cu(S0), H=x["H"], G=x["G"],
                                  decay_kind=x["decay_kind"], scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return (None if o is None else o.cpu().numpy()), (None if S is None else S.cpu().numpy())


def ref(x, S0=None):
    return oracle.recur_diag(*(x[n].numpy() for n in ("q", "k", "v", "d")),
                             None if S0 is None else S0.numpy().astype(np.float64),
                             H=x["H"], G=x["G"], decay_kind=x["decay_kind"], scale=x["scale"])


# ------------------------------------------------------------------ parity
@pytest.mark.parametrize("kind,G", [("gla", None), ("mamba2", 1), ("mamba2", 2)])
@pytest.mark.parametrize("dv", [128, 64])
@pytest.mark.parametrize("T", [1, 5, 127, 128, 129, 300])
def test_parity_small(ctx, kind, G, dv, T):
    B, H = 2, 4
    x = make(kind, B, T, H, dv, G=G, seed=T % 5)
    S0 = synth.normal((B, H, 128, dv), 7000 + T) * 0.5
    o, S = run_chunked(ctx, x, S0)
    ro, rS = ref(x, S0)
    assert _nrel(o, ro) <= TOL
    assert _nrel(S, rS) <= TOL


@pytest.mark.parametrize("kind", ["gla", "mamba2"])
def test_zero_initial_state_and_optional_outputs(ctx, kind):
    B, T, H, dv = 1, 260, 2, 128
    x = make(kind, B, T, H, dv, seed=3)
    ro, rS = ref(x)
    o, S = run_chunked(ctx, x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL
    o2, S2 = run_chunked(ctx, x, o=False)
    assert o2 is None and np.array_equal(S2, S)
    o3, S3 = run_chunked(ctx, x, S_out=False)
    assert S3 is None and np.array_equal(o3, o)


@pytest.mark.parametrize("kind", ["gla", "mamba2"])
def test_unit_decay_is_causal_linear_attention(ctx, kind):
    """d = 1: o_t = scale * sum_{j <= t} (q_t . k_j) v_j (every pair weight 1)."""
    B, T, H, dv = 1, 200, 2, 64
    x = make(kind, B, T, H, dv, seed=1)
    x = dict(x, d=torch.ones_like(x["d"]))
    o, S = run_chunked(ctx, x)
    ro, rS = ref(x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL


def test_strong_per_head_decay_has_no_range_limit(ctx, sr):
    """Per-head decays apply the exact pair weight, so a decay product far
    below 2^-60 inside one chunk is still computed (and the state forgets)."""
    B, T, H, dv = 1, 256, 2, 64
    x = make("mamba2", B, T, H, dv, seed=2)
    x = dict(x, d=torch.full_like(x["d"], 0.25))
    o, S = run_chunked(ctx, x)
    ro, rS = ref(x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL


# ------------------------------------------------------------------ splits
@pytest.mark.parametrize("kind", ["gla", "mamba2"])
@pytest.mark.parametrize("split", [CHUNK, 3 * CHUNK])
def test_split_at_chunk_multiple_is_bit_exact(ctx, kind, split):
    B, T, H, dv = 2, 700, 2, 128
    x = make(kind, B, T, H, dv, seed=4)
    S0 = synth.normal((B, H, 128, dv), 7100) * 0.5
    o, S = run_chunked(ctx, x, S0)
    first = {n: (x[n][:, :split].contiguous() if n in ("q", "k", "v", "d") else x[n]) for n in x}
    rest = {n: (x[n][:, split:].contiguous() if n in ("q", "k", "v", "d") else x[n]) for n in x}
    o1, S1 = run_chunked(ctx, first, S0)
    o2, S2 = run_chunked(ctx, rest, torch.from_numpy(S1))
    assert np.array_equal(np.concatenate([o1, o2], axis=1), o)
    assert np.array_equal(S2, S)


def test_split_off_the_chunk_grid_stays_within_tolerance(ctx):
    B, T, H, dv = 1, 500, 2, 128
    x = make("gla", B, T, H, dv, seed=0)
    split = 200
    first = {n: (x[n][:, :split].contiguous() if n in ("q", "k", "v", "d") else x[n]) for n in x}
    rest = {n: (x[n][:, split:].contiguous() if n in ("q", "k", "v", "d") else x[n]) for n in x}
    _, S1 = run_chunked(ctx, first)
    o2, S2 = run_chunked(ctx, rest, torch.from_numpy(S1))
    ro, rS = ref(x)
    assert _nrel(o2, ro[:, split:]) <= TOL and _nrel(S2, rS) <= TOL


# ------------------------------------------------------------------ full size
@pytest.mark.parametrize("name", ["gla", "mamba2"])
def test_full_size_sampled_heads(ctx, name):
    """The full workloads in the launch configuration the benchmark times;
    sampled (b, h) sequences recomputed one by one by the oracle."""
    x = synth.config_inputs(name)
    c = synth.CONFIGS[name]
    B, H = c["B"], c["H"]
    o, S = run_chunked(ctx, x)
    rng = np.random.default_rng(31)
    heads = sorted({(int(rng.integers(B)), int(rng.integers(H))) for _ in range(3)} | {(0, 0), (B - 1, H - 1)})
    for (b, h) in heads:
        g = h // (H // x["G"])
        xs = dict(x, q=x["q"][b:b + 1, :, g:g + 1].contiguous(), k=x["k"][b:b + 1, :, g:g + 1].contiguous(),
                  v=x["v"][b:b + 1, :, h:h + 1].contiguous(), d=x["d"][b:b + 1, :, h:h + 1].contiguous(), H=1, G=1)
        ro, rS = ref(xs)
        assert _nrel(o[b:b + 1, :, h:h + 1], ro) <= TOL
        assert _nrel(S[b:b + 1, h:h + 1], rS) <= TOL


# ------------------------------------------------------------------ strong per-key decays
def _strong(x, mode, seed):
    """Per-key decays whose in-chunk products leave the single-anchor range:
    d = 2^-4 at every token, GLA decays exp(logsigmoid(N(0,1))) without the
    /16 (a product of about 2^-74 over half a chunk), or chunks that
    alternate between the workload's mild decays and 2^-4 (flagged and
    unflagged chunks in one call)."""
    d = x["d"]
    if mode == "pow2":
        d = torch.full_like(d, 2.0 ** -4)
    elif mode == "logsigmoid":
        d = torch.exp(torch.nn.functional.logsigmoid(synth.normal(tuple(d.shape), 9900 + seed)))
    else:
        d = d.clone()
        for n0 in range(CHUNK, d.shape[1], 2 * CHUNK):
            d[:, n0:n0 + CHUNK] = 2.0 ** -4
    return dict(x, d=d.contiguous())


@pytest.mark.parametrize("mode", ["pow2", "logsigmoid", "mixed"])
@pytest.mark.parametrize("dv", [128, 64])
@pytest.mark.parametrize("T", [128, 300, 640])
def test_strong_per_key_decays_within_tolerance(ctx, mode, dv, T):
    """Chunks beyond the single-anchor range are evaluated step by step from
    their start state: within the chunked form's tolerance of the fp64
    oracle, with a start state, and no error recorded."""
    B, H = 2, 3
    x = _strong(make("gla", B, T, H, dv, seed=T % 5), mode, T)
    S0 = synth.normal((B, H, 128, dv), 9950 + T) * 0.5
    o, S = run_chunked(ctx, x, S0)
    ro, rS = ref(x, S0)
    assert _nrel(o, ro) <= TOL
    assert _nrel(S, rS) <= TOL


@pytest.mark.parametrize("mode", ["pow2", "mixed"])
def test_strong_gated_per_key_decays(ctx, mode):
    B, T, H, dv = 2, 300, 2, 128
    x = synth.gated_memory_inputs(B, T, H, 128, dv, per_key=True, cid=360)
    x = _strong(x, mode, 7)
    o, S = run_chunked(ctx, x)
    ro, rS = ref(x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL


def test_strong_decays_split_at_chunk_multiple_bit_exact(ctx):
    """The flagged chunks' step-by-step outputs depend only on the chunk's
    start state and its tokens, so splits at chunk multiples stay bit-exact."""
    B, T, H, dv = 1, 512, 2, 64
    x = _strong(make("gla", B, T, H, dv, seed=3), "mixed", 11)
    o, S = run_chunked(ctx, x)
    cut = 2 * CHUNK
    x1 = {k: (v[:, :cut].contiguous() if torch.is_tensor(v) and v.dim() == 4 else v) for k, v in x.items()}
    x2 = {k: (v[:, cut:].contiguous() if torch.is_tensor(v) and v.dim() == 4 else v) for k, v in x.items()}
    o1, S1 = run_chunked(ctx, x1)
    o2, S2 = run_chunked(ctx, x2, torch.from_numpy(S1))
    assert np.array_equal(np.concatenate([o1, o2], axis=1), o) and np.array_equal(S2, S)


# ------------------------------------------------------------------ errors
def test_non_positive_decay_is_reported(ctx, sr):
    B, T, H, dv = 1, 128, 1, 64
    x = make("gla", B, T, H, dv, seed=0)
    d = x["d"].clone()
    d[0, 5, 0, 17] = 0.0
    run_chunked(ctx, dict(x, d=d))
    assert ctx.last_error() == sr.SN_E_RANGE
    assert ctx.last_error() == sr.SN_OK                    # read once, cleared


@pytest.mark.parametrize("per_key", [True, False])
@pytest.mark.parametrize("dv", [128, 64])
@pytest.mark.parametrize("T", [5, 128, 300])
@pytest.mark.parametrize("with_state", [False, True])
def test_gated_parity(ctx, per_key, dv, T, with_state):
    """Gated injection S = p (.) S + (1 - p) (.) (k v^T): the diagonal
    recurrence with keys weighted by 1 - p, which every kernel of the chunked
    form applies where it scales the keys (per-head gates with dv = 64 run the
    block-of-heads kernels)."""
    B, H = 2, 3
    x = synth.gated_memory_inputs(B, T, H, 128, dv, per_key=per_key, cid=340 + T % 5)
    S0 = synth.normal((B, H, 128, dv), 9700 + T) * 0.5 if with_state else None
    o, S = run_chunked(ctx, x, S0)
    ro, rS = ref(x, S0)
    assert _nrel(o, ro) <= TOL
    assert _nrel(S, rS) <= TOL


def test_gated_per_head_blocks_sharing_one_group(ctx):
    """Per-head gates with grouped keys: the output kernel weights each head's
    copy of Q K^T by that head's decays and gates (two heads per CTA here)."""
    B, T, H, G, dv = 4, 2048, 8, 2, 64
    x = synth.mamba2_inputs(B, T, H, G, 128, dv, cid=350)
    x = dict(x, decay_kind=synth.DECAY_PER_HEAD_GATED)
    S0 = synth.normal((B, H, 128, dv), 9800) * 0.5
    o, S = run_chunked(ctx, x, S0)
    per = H // G
    for b in (0, B - 1):
        for h in range(H):
            g = h // per
            xs = dict(x, q=x["q"][b:b + 1, :, g:g + 1].contiguous(), k=x["k"][b:b + 1, :, g:g + 1].contiguous(),
                      v=x["v"][b:b + 1, :, h:h + 1].contiguous(), d=x["d"][b:b + 1, :, h:h + 1].contiguous(),
                      H=1, G=1)
            ro, rS = ref(xs, S0[b:b + 1, h:h + 1].contiguous())
            assert _nrel(o[b:b + 1, :, h:h + 1], ro) <= TOL, (b, h)
            assert _nrel(S[b:b + 1, h:h + 1], rS) <= TOL, (b, h)


@pytest.mark.parametrize("kind", ["gla", "mamba2"])
def test_zero_decay_is_reported(ctx, sr, kind):
    B, T, H, dv = 1, 64, 1, 64
    x = make(kind, B, T, H, dv, seed=0)
    d = x["d"].clone()
    d[0, 10] = 0.0
    run_chunked(ctx, dict(x, d=d))
    assert ctx.last_error() == sr.SN_E_RANGE


def test_unsupported_shapes_and_missing_workspace(ctx, sr):
    abi = sr._abi
    x = make("gla", 1, 16, 1, 64, seed=0)
    q, k, v, d = (cu(x[n]) for n in ("q", "k", "v", "d"))
    o = torch.empty((1, 16, 1, 64), device="cuda")
    S = torch.empty((1, 1, 128, 64), device="cuda")
    # no workspace yet on this context
    assert abi.sn_recur_diag_chunked(ctx.handle, 1, 16, 1, 1, 128, 64, sr.SN_DECAY_PER_KEY, 1.0, q, k, v, d,
                                     None, S, o) == sr.SN_E_NOMEM
    ctx.ensure_workspace_bytes(abi.sn_recur_chunked_workspace_bytes(1, 16, 1, 128, 64))
    assert abi.sn_recur_diag_chunked(ctx.handle, 1, 16, 1, 1, 128, 64, 7, 1.0, q, k, v, d,
                                     None, S, o) == sr.SN_E_INVAL
    x64 = synth.gla_inputs(1, 16, 1, 64, 64, cid=320)
    q6, k6, v6, d6 = (cu(x64[n]) for n in ("q", "k", "v", "d"))
    S6 = torch.empty((1, 1, 64, 64), device="cuda")
    assert abi.sn_recur_diag_chunked(ctx.handle, 1, 16, 1, 1, 64, 64, sr.SN_DECAY_PER_KEY, 1.0, q6, k6, v6, d6,
                                     None, S6, o) == sr.SN_E_UNSUPPORTED
    torch.cuda.synchronize()
    assert abi.sn_recur_chunked_workspace_bytes(0, 16, 1, 128, 64) == -1


def test_lookback_scan_after_chunked_call_on_same_context(ctx, sr):
    """The chunk states overwrite the workspace; the next look-back scan must
    clear its flag area again and stay bit-exact with the sequential kernel."""
    x = make("gla", 1, 300, 2, 128, seed=0)
    run_chunked(ctx, x)
    s = synth.scan_inputs(2, 2048, 64, large=True)
    a, b, s0 = cu(s["a"]), cu(s["b"]), cu(s["s0"])
    ref_out, ref_fin = ctx.scan_fma(a, b, s0)
    ctx.ensure_workspace(2, 2048, 64)
    run_chunked(ctx, x)                                     # dirty the (now larger) workspace again
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
    out, fin = ctx.scan_fma(a, b, s0)
    torch.cuda.synchronize()
    ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
    # the look-back kernel is deterministic; compare with the sequential kernel within 1e-5
    assert _nrel(out.cpu().numpy(), ref_out.cpu().numpy()) <= 1e-5
    assert _nrel(fin.cpu().numpy(), ref_fin.cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("G", [1, 2])
def test_head_blocks_sharing_one_group(ctx, G):
    """Per-head decays with many heads per group: the output kernel forms Q K^T
    once per block of heads (4 heads per CTA at this size); every head of two
    batch rows is checked against the oracle."""
    B, T, H, dv = 4, 2048, 24, 64
    x = synth.mamba2_inputs(B, T, H, G, 128, dv, cid=330 + G)
    S0 = synth.normal((B, H, 128, dv), 7200 + G) * 0.5
    o, S = run_chunked(ctx, x, S0)
    per = H // G
    for b in (0, B - 1):
        for h in range(H):
            g = h // per
            xs = dict(x, q=x["q"][b:b + 1, :, g:g + 1].contiguous(), k=x["k"][b:b + 1, :, g:g + 1].contiguous(),
                      v=x["v"][b:b + 1, :, h:h + 1].contiguous(), d=x["d"][b:b + 1, :, h:h + 1].contiguous(),
                      H=1, G=1)
            ro, rS = ref(xs, S0[b:b + 1, h:h + 1].contiguous())
            assert _nrel(o[b:b + 1, :, h:h + 1], ro) <= TOL, (b, h)
            assert _nrel(S[b:b + 1, h:h + 1], rS) <= TOL, (b, h)


@pytest.mark.parametrize("kind", ["gla", "mamba2"])
def test_in_place_state(ctx, kind):
    """S_in and S_out may be the same buffer (continuation in place)."""
    B, T, H, dv = 2, 300, 2, 128
    x = make(kind, B, T, H, dv, seed=1)
    S0 = synth.normal((B, H, 128, dv), 7300) * 0.5
    o_ref, S_ref = run_chunked(ctx, x, S0)
    Sd = S0.cuda()
    o, S = ctx.recur_diag_chunked(*(cu(x[n]) for n in ("q", "k", "v", "d")), Sd, H=x["H"], G=x["G"],
                                  decay_kind=x["decay_kind"], scale=x["scale"], S_out=Sd)
    torch.cuda.synchronize()
    assert S.data_ptr() == Sd.data_ptr()
    assert np.array_equal(Sd.cpu().numpy(), S_ref) and np.array_equal(o.cpu().numpy(), o_ref)


def test_grouped_keys_with_per_key_decay(ctx):
    """Per-key decays with q, k shared by groups of heads (G < H)."""
    B, T, H, G, dv = 2, 260, 4, 2, 64
    x = make("gla", B, T, H, dv, seed=2)
    q = synth.normal((B, T, G, 128), 7400) * 0.088
    k = synth.normal((B, T, G, 128), 7401) * 0.088
    x = dict(x, q=q, k=k, G=G)
    o, S = run_chunked(ctx, x)
    ro, rS = ref(x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL
