"""GPU parity of the chunked tensor-core delta rule (sn_recur_delta_chunked)
against the fp64 oracle.

Bar: o and the final state within 2e-3 normwise of the fp64 oracle (tf32
operands, as for the chunked diagonal-decay form); splits at multiples of the
128-token chunk bit-exact within the GPU path; beta = 1 with unit keys keeps
the retrieval identity S_t^T k_t = v_t that the oracle's pins fix.
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


def run(ctx, x, S0=None, **kw):
    o, S = ctx.recur_delta_chunked(*(cu(x[n]) for n in ("q", "k", "v", "beta")), cu(S0), scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return (None if o is None else o.cpu().numpy()), (None if S is None else S.cpu().numpy())


def ref(x, S0=None):
    return oracle.recur_delta(*(x[n].numpy() for n in ("q", "k", "v", "beta")),
                              None if S0 is None else S0.numpy().astype(np.float64), scale=x["scale"])


@pytest.mark.parametrize("T", [1, 5, 127, 128, 129, 300, 640])
@pytest.mark.parametrize("with_state", [False, True])
def test_parity(ctx, T, with_state):
    B, H = 2, 3
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=400 + T % 7)
    S0 = synth.normal((B, H, 128, 128), 8000 + T) * 0.5 if with_state else None
    o, S = run(ctx, x, S0)
    ro, rS = ref(x, S0)
    assert _nrel(o, ro) <= TOL
    assert _nrel(S, rS) <= TOL


def test_unit_beta_retrieves_the_value(ctx):
    """beta = 1 and |k| = 1: S_t^T k_t = v_t after every step, so the last
    token's key reads back its value from the final state."""
    B, T, H = 1, 200, 2
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=410)
    x = dict(x, beta=torch.ones_like(x["beta"]))
    _, S = run(ctx, x)
    k_last = x["k"][:, -1].numpy().astype(np.float64)           # (B, H, dk)
    got = np.einsum("bhij,bhi->bhj", S.astype(np.float64), k_last)
    assert _nrel(got, x["v"][:, -1].numpy()) <= TOL


@pytest.mark.parametrize("split", [CHUNK, 2 * CHUNK])
def test_split_at_chunk_multiple_is_bit_exact(ctx, split):
    B, T, H = 2, 600, 2
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=420)
    S0 = synth.normal((B, H, 128, 128), 8100) * 0.5
    o, S = run(ctx, x, S0)
    first = {n: (x[n][:, :split].contiguous() if n in ("q", "k", "v", "beta") else x[n]) for n in x}
    rest = {n: (x[n][:, split:].contiguous() if n in ("q", "k", "v", "beta") else x[n]) for n in x}
    o1, S1 = run(ctx, first, S0)
    o2, S2 = run(ctx, rest, torch.from_numpy(S1))
    assert np.array_equal(np.concatenate([o1, o2], axis=1), o)
    assert np.array_equal(S2, S)


def test_optional_outputs(ctx):
    x = synth.deltanet_inputs(1, 300, 2, 128, 128, cid=430)
    o, S = run(ctx, x)
    o2, S2 = run(ctx, x, o=False)
    assert o2 is None and np.array_equal(S2, S)
    o3, S3 = run(ctx, x, S_out=False)
    assert S3 is None and np.array_equal(o3, o)


def test_full_size_sampled_heads(ctx):
    """The full DeltaNet workload (B4 T4096 H8 128x128) in the launch
    configuration the benchmark times; sampled heads recomputed by the oracle."""
    x = synth.config_inputs("deltanet")
    o, S = run(ctx, x)
    rng = np.random.default_rng(41)
    heads = sorted({(int(rng.integers(4)), int(rng.integers(8))) for _ in range(3)} | {(0, 0), (3, 7)})
    for (b, h) in heads:
        xs = {n: x[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "beta")}
        xs["scale"] = x["scale"]
        ro, rS = ref(xs)
        assert _nrel(o[b:b + 1, :, h:h + 1], ro) <= TOL
        assert _nrel(S[b:b + 1, h:h + 1], rS) <= TOL


def test_unsupported_and_missing_workspace(ctx, sr):
    abi = sr._abi
    x = synth.deltanet_inputs(1, 16, 1, 64, 64, cid=440)
    q, k, v, beta = (cu(x[n]) for n in ("q", "k", "v", "beta"))
    o = torch.empty((1, 16, 1, 64), device="cuda")
    assert abi.sn_recur_delta_chunked(ctx.handle, 1, 16, 1, 64, 64, 1.0, q, k, v, beta, None, None, o) == \
        sr.SN_E_UNSUPPORTED
    x = synth.deltanet_inputs(1, 16, 1, 128, 128, cid=441)
    q, k, v, beta = (cu(x[n]) for n in ("q", "k", "v", "beta"))
    o = torch.empty((1, 16, 1, 128), device="cuda")
    assert abi.sn_recur_delta_chunked(ctx.handle, 1, 16, 1, 128, 128, 1.0, q, k, v, beta, None, None, o) == \
        sr.SN_E_NOMEM
    assert abi.sn_recur_delta_chunked_workspace_bytes(1, 0, 1, 128, 128) == -1
    torch.cuda.synchronize()


def test_in_place_state(ctx):
    x = synth.deltanet_inputs(2, 300, 2, 128, 128, cid=450)
    S0 = synth.normal((2, 2, 128, 128), 8200) * 0.5
    o_ref, S_ref = run(ctx, x, S0)
    Sd = S0.cuda()
    o, S = ctx.recur_delta_chunked(*(cu(x[n]) for n in ("q", "k", "v", "beta")), Sd, scale=x["scale"], S_out=Sd)
    torch.cuda.synchronize()
    assert S.data_ptr() == Sd.data_ptr()
    assert np.array_equal(Sd.cpu().numpy(), S_ref) and np.array_equal(o.cpu().numpy(), o_ref)


@pytest.mark.parametrize("segments", [2, 3, 4, 8, 0])
def test_segments_give_the_same_bits(ctx, sr, segments):
    """The pipelined call (segments of chunks over side streams) against one
    segment: the state crosses segments in fp32, so the bits must agree.  T =
    1100 leaves a ragged last chunk of 76 tokens."""
    B, T, H = 2, 1100, 3
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=460)
    S0 = synth.normal((B, H, 128, 128), 8300) * 0.5
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 1)
    o1, S1 = run(ctx, x, S0)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, segments)
    assert ctx.get_option(sr.SN_OPT_DELTA_SEGMENTS) == segments
    o, S = run(ctx, x, S0)
    assert np.array_equal(o, o1) and np.array_equal(S, S1)
    _, S_only = run(ctx, x, S0, o=False)
    assert np.array_equal(S_only, S1)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)


def test_fused_on_the_deltanet_workload_gives_the_same_bits(ctx, sr):
    """The default call on the DeltaNet workload shape (B4 T4096 H8: one
    cooperative launch of preparation and chains, then the output stage)
    against one pipelined segment, bit for bit."""
    B, T, H = 4, 4096, 8
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=470)
    S0 = synth.normal((B, H, 128, 128), 8310) * 0.5
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 1)
    o1, S1 = run(ctx, x, S0)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)
    o, S = run(ctx, x, S0)
    assert np.array_equal(o, o1) and np.array_equal(S, S1)


def test_many_heads_fall_back_to_the_pipeline(ctx, sr):
    """B*H above half the SMs: the default call takes the segmented pipeline
    and still gives the bits of one segment."""
    B, T, H = 8, 300, 10
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=480)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 1)
    o1, S1 = run(ctx, x)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)
    o, S = run(ctx, x)
    assert np.array_equal(o, o1) and np.array_equal(S, S1)


def test_fused_bounded_wait_reports_timeout(ctx, sr):
    """The chains of the fused call wait for a ready value no CTA writes: each
    wait runs out after the limit, the kernel returns, the context reports
    SN_E_TIMEOUT once, and the next call is exact again."""
    B, T, H = 1, 640, 2
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=490)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)
    ctx.set_option(sr.SN_OPT_WAIT_LIMIT_US, 2000)
    ctx.set_option(sr.SN_OPT_DEBUG_POISON, 1)
    run(ctx, x)
    assert ctx.last_error() == sr.SN_E_TIMEOUT
    assert ctx.last_error() == sr.SN_OK             # cleared
    ctx.set_option(sr.SN_OPT_DEBUG_POISON, 0)
    o, S = run(ctx, x)
    assert ctx.last_error() == sr.SN_OK
    ro, rS = ref(x)
    assert _nrel(o, ro) <= TOL and _nrel(S, rS) <= TOL


def test_fused_replayed_from_a_cuda_graph(ctx, sr):
    """The default one-launch call captured in a CUDA graph (with the memset
    that clears its control words) and replayed on new inputs: each replay
    equals an uncaptured call bit for bit."""
    B, T, H = 2, 1100, 3
    ins = [synth.deltanet_inputs(B, T, H, 128, 128, cid=500 + i) for i in range(2)]
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)
    expect = [run(ctx, x) for x in ins]
    d = {n: ins[0][n].cuda().clone() for n in ("q", "k", "v", "beta")}
    o = torch.empty((B, T, H, 128), device="cuda")
    S = torch.empty((B, H, 128, 128), device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = sr.sn_recur_delta_chunked(ctx.handle, B, T, H, 128, 128, ins[0]["scale"], d["q"], d["k"], d["v"],
                                       d["beta"], None, S, o, torch.cuda.current_stream())
    assert st == sr.SN_OK
    for _ in range(2):
        for x, (eo, eS) in zip(ins, expect):
            assert x["scale"] == ins[0]["scale"]
            for n in d:
                d[n].copy_(x[n])
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(o.cpu().numpy(), eo) and np.array_equal(S.cpu().numpy(), eS)


def test_segments_in_place_on_a_side_stream(ctx, sr):
    """Pipelined call issued on a non-default stream, state in place: the
    results are ordered on that stream."""
    B, T, H = 1, 1300, 2
    x = synth.deltanet_inputs(B, T, H, 128, 128, cid=470)
    S0 = synth.normal((B, H, 128, 128), 8400) * 0.5
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 1)
    o_ref, S_ref = run(ctx, x, S0)
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 4)
    side = torch.cuda.Stream()
    ins = [cu(x[n]) for n in ("q", "k", "v", "beta")]
    Sd = S0.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        o, S = ctx.recur_delta_chunked(*ins, Sd, scale=x["scale"], S_out=Sd, stream=side)
        o_host = o.to("cpu", non_blocking=False)
        S_host = Sd.to("cpu", non_blocking=False)
    torch.cuda.synchronize()
    ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, 0)
    assert np.array_equal(o_host.numpy(), o_ref) and np.array_equal(S_host.numpy(), S_ref)


def test_segment_option_range(ctx, sr):
    for bad in (-1, 9):
        with pytest.raises(sr.SnError):
            ctx.set_option(sr.SN_OPT_DELTA_SEGMENTS, bad)
    assert ctx.get_option(sr.SN_OPT_DELTA_SEGMENTS) == 0
