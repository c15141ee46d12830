"""Pins of the CPU oracle's matrix-state recurrences.

Sources: "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
§4 (segment continuation), §4.1 (Mamba-2 scalar decay, grouped B/C), §4.2
(DeltaNet rank-1 form and its explicit (I - b k k^T) S + b k v^T twin, with
the warning that a wrong-side multiply is silent when dk == dv), §4.3 (GLA
decay decomposes elementwise; readout S^T q * scale), §5.1 (RWKV-7 rank-1
removal), and "我拿同一份权重和 llama.cpp 正面比了一场：我手写的 C 内核，慢了
1.1–1.7 倍" §3 (the per-head value-slice bug that only shows when dk != dv).

Checks use explicit matrix products (numpy matmul as the library primitive),
brute-force unrolled products on T <= 6, special cases with closed forms,
bitwise decompositions into the already-pinned scan, and hand fixtures.
"""
import numpy as np
import pytest

import oracle
from tests import _golden


def _rng(seed):
    return np.random.default_rng(seed)


def _sig(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def _l2n(x):
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def _outer(x, y):
    """Outer product in fp64 (inputs widened before multiplying)."""
    return np.outer(np.asarray(x, np.float64), np.asarray(y, np.float64))


def _nrel(x, r):
    return float(np.max(np.abs(np.asarray(x, np.float64) - r)) / max(np.max(np.abs(r)), 1e-300))


# ------------------------------------------------------------------ fixtures
@pytest.mark.parametrize("prec", ["f64", "f32"])
@pytest.mark.parametrize("name", ["diag_gla_dyadic.txt", "diag_mamba2_dyadic.txt"])
def test_diag_hand_fixture(name, prec):
    g = _golden.load(name)
    B, T, H, G, dk, dv = g["shape"]
    kind = int(g["decay_kind"][0])
    dshape = (B, T, H, dk) if kind == oracle.DECAY_PER_KEY else (B, T, H)
    o, S = oracle.recur_diag(_golden.f32(g["q"], (B, T, G, dk)), _golden.f32(g["k"], (B, T, G, dk)),
                             _golden.f32(g["v"], (B, T, H, dv)), _golden.f32(g["d"], dshape),
                             H=H, G=G, decay_kind=kind, scale=g["scale"][0], prec=prec)
    assert np.array_equal(o, np.asarray(g["o"]).reshape(B, T, H, dv))
    assert np.array_equal(S, np.asarray(g["S"]).reshape(B, H, dk, dv))


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_delta_hand_fixture(prec):
    g = _golden.load("delta_dyadic.txt")
    B, T, H, dk, dv = g["shape"]
    o, S = oracle.recur_delta(_golden.f32(g["q"], (B, T, H, dk)), _golden.f32(g["k"], (B, T, H, dk)),
                              _golden.f32(g["v"], (B, T, H, dv)), _golden.f32(g["beta"], (B, T, H)),
                              np.asarray(g["S0"]).reshape(B, H, dk, dv), scale=g["scale"][0], prec=prec)
    assert np.array_equal(o, np.asarray(g["o"]).reshape(B, T, H, dv))
    assert np.array_equal(S, np.asarray(g["S"]).reshape(B, H, dk, dv))


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_rwkv7_hand_fixture(prec):
    g = _golden.load("rwkv7_dyadic.txt")
    B, T, H, dk, dv = g["shape"]
    o, S = oracle.recur_rwkv7(_golden.f32(g["q"], (B, T, H, dk)), _golden.f32(g["k"], (B, T, H, dk)),
                              _golden.f32(g["v"], (B, T, H, dv)), _golden.f32(g["w"], (B, T, H, dk)),
                              np.asarray(g["S0"]).reshape(B, H, dv, dk), prec=prec)
    assert np.array_equal(o, np.asarray(g["o"]).reshape(B, T, H, dv))
    assert np.array_equal(S, np.asarray(g["S"]).reshape(B, H, dv, dk))


# ------------------------------------------------------------------ inputs
def _diag_inputs(seed, B, T, H, G, dk, dv, per_key=True):
    rng = _rng(seed)
    q = (rng.standard_normal((B, T, G, dk)) / np.sqrt(dk)).astype(np.float32)
    k = (rng.standard_normal((B, T, G, dk)) / np.sqrt(dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    if per_key:
        d = np.exp(np.log(_sig(rng.standard_normal((B, T, H, dk)))) / 16).astype(np.float32)
    else:
        d = _sig(rng.standard_normal((B, T, H)) + 2)
    S0 = rng.standard_normal((B, H, dk, dv))
    return q, k, v, d, S0


def _delta_inputs(seed, B, T, H, dk, dv):
    rng = _rng(seed)
    q = _l2n(rng.standard_normal((B, T, H, dk)))
    k = _l2n(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    beta = _sig(rng.standard_normal((B, T, H)))
    S0 = rng.standard_normal((B, H, dk, dv))
    return q, k, v, beta, S0


def _rwkv_inputs(seed, B, T, H, dk, dv):
    rng = _rng(seed)
    w = np.exp(-np.exp(rng.normal(-0.5, 0.5, (B, T, H, dk)))).astype(np.float32)
    k = _l2n(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    S0 = rng.standard_normal((B, H, dv, dk))
    return q, k, v, w, S0


# ------------------------------------------------------------------ diag
def test_diag_explicit_diagonal_matrix_product():
    """GLA decay as a full dk x dk diagonal matrix times S, plus the outer
    product, matches the rowwise-scaled update (fp64)."""
    B, T, H, dk, dv = 2, 24, 3, 8, 5
    q, k, v, d, S0 = _diag_inputs(10, B, T, H, H, dk, dv)
    o, S = oracle.recur_diag(q, k, v, d, S0, H=H, G=H, decay_kind=0, scale=0.3)
    for b in range(B):
        for h in range(H):
            M = S0[b, h].copy()
            for t in range(T):
                M = np.diag(d[b, t, h].astype(np.float64)) @ M + _outer(k[b, t, h], v[b, t, h])
                assert _nrel(o[b, t, h], 0.3 * (M.T @ q[b, t, h].astype(np.float64))) < 1e-13
            assert _nrel(S[b, h], M) < 1e-13


def test_diag_bruteforce_unrolled():
    """T <= 6: S_T = (prod D_t) S0 + sum_j (prod_{t>j} D_t) k_j v_j^T."""
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    q, k, v, d, S0 = _diag_inputs(11, B, T, H, H, dk, dv)
    _, S = oracle.recur_diag(q, k, v, d, S0, H=H, G=H, decay_kind=0, scale=1.0)
    for h in range(H):
        D = [np.diag(d[0, t, h].astype(np.float64)) for t in range(T)]
        acc = np.eye(dk)
        for t in range(T):
            acc = D[t] @ acc
        ref = acc @ S0[0, h]
        for j in range(T):
            P = np.eye(dk)
            for t in range(j + 1, T):
                P = D[t] @ P
            ref = ref + P @ _outer(k[0, j, h], v[0, j, h])
        assert _nrel(S[0, h], ref) < 1e-13


def test_diag_no_decay_is_causal_linear_attention():
    """d = 1: o_t = scale * sum_{j<=t} (k_j . q_t) v_j, i.e. the masked product
    scale * tril(Q K^T) V."""
    B, T, H, dk, dv = 1, 40, 2, 16, 8
    q, k, v, _, _ = _diag_inputs(12, B, T, H, H, dk, dv)
    d = np.ones((B, T, H, dk), np.float32)
    o, _ = oracle.recur_diag(q, k, v, d, None, H=H, G=H, decay_kind=0, scale=0.5)
    for h in range(H):
        Q, K, V = (x[0, :, h].astype(np.float64) for x in (q, k, v))
        ref = 0.5 * np.tril(Q @ K.T) @ V
        assert _nrel(o[0, :, h], ref) < 1e-13


def test_diag_full_decay_keeps_only_last_outer_product():
    """d = 0: S_t = k_t v_t^T, so o_t = scale (k_t . q_t) v_t."""
    B, T, H, dk, dv = 1, 10, 1, 8, 4
    q, k, v, _, S0 = _diag_inputs(13, B, T, H, H, dk, dv)
    d = np.zeros((B, T, H, dk), np.float32)
    o, S = oracle.recur_diag(q, k, v, d, S0, H=H, G=H, decay_kind=0, scale=2.0)
    for t in range(T):
        ref = 2.0 * float(k[0, t, 0].astype(np.float64) @ q[0, t, 0]) * v[0, t, 0].astype(np.float64)
        assert _nrel(o[0, t, 0], ref) < 1e-14
    assert _nrel(S[0, 0], _outer(k[0, -1, 0], v[0, -1, 0])) < 1e-15


@pytest.mark.parametrize("per_key", [True, False])
def test_diag_f32_decomposes_into_fma_scans(per_key):
    """Every state entry is an independent FMA-form scan with a = d_i (or the
    head's scalar dA) and b = fl(k_i v_j) -- bitwise in fp32 ("SunnyNet
    工程化实录" §4.1 and §4.3: the decay decomposes elementwise)."""
    B, T, H, dk, dv = 1, 50, 2, 8, 4
    q, k, v, d, S0 = _diag_inputs(14, B, T, H, H, dk, dv, per_key=per_key)
    S0 = S0.astype(np.float32)
    _, S = oracle.recur_diag(q, k, v, d, S0, H=H, G=H, decay_kind=0 if per_key else 1,
                             scale=1.0, prec="f32")
    for h in range(H):
        if per_key:
            a = np.repeat(d[0, :, h, :, None], dv, axis=2)
        else:
            a = np.broadcast_to(d[0, :, h, None, None], (T, dk, dv))
        bb = (k[0, :, h, :, None] * v[0, :, h, None, :]).astype(np.float32)
        _, sf = oracle.scan_fma(np.ascontiguousarray(a.reshape(1, T, dk * dv)),
                                np.ascontiguousarray(bb.reshape(1, T, dk * dv)),
                                S0[0, h].reshape(1, dk * dv), prec="f32")
        assert np.array_equal(sf.reshape(dk, dv).view(np.uint32), S[0, h].view(np.uint32))


def test_diag_groups_equal_replicated_heads():
    """G < H: head h reads group h // (H // G); same as G = H with k, q
    replicated per head (bitwise)."""
    B, T, H, G, dk, dv = 2, 12, 6, 2, 8, 4
    q, k, v, _, S0 = _diag_inputs(15, B, T, H, G, dk, dv)
    d = _sig(_rng(16).standard_normal((B, T, H)) + 2)
    o1, S1 = oracle.recur_diag(q, k, v, d, S0, H=H, G=G, decay_kind=1, scale=1.0)
    rep = np.repeat(np.arange(G), H // G)
    o2, S2 = oracle.recur_diag(np.ascontiguousarray(q[:, :, rep]), np.ascontiguousarray(k[:, :, rep]),
                               v, d, S0, H=H, G=H, decay_kind=1, scale=1.0)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)
    # and a wrong group map (h % G) gives a different answer
    rep_bad = np.arange(H) % G
    o3, _ = oracle.recur_diag(np.ascontiguousarray(q[:, :, rep_bad]), np.ascontiguousarray(k[:, :, rep_bad]),
                              v, d, S0, H=H, G=H, decay_kind=1, scale=1.0)
    assert not np.allclose(o1, o3)


@pytest.mark.parametrize("fn", ["diag", "delta", "rwkv7"])
def test_head_value_slices_are_independent(fn):
    """dk != dv and distinct per-head values: perturbing head 1's v changes only
    head 1's outputs (the per-head value-slice bug of the llama.cpp comparison
    article §3 would leak it into the other heads)."""
    B, T, H, dk, dv = 1, 9, 3, 8, 5
    if fn == "diag":
        q, k, v, d, S0 = _diag_inputs(17, B, T, H, H, dk, dv)
        run = lambda vv: oracle.recur_diag(q, k, vv, d, S0, H=H, G=H, decay_kind=0, scale=1.0)
    elif fn == "delta":
        q, k, v, beta, S0 = _delta_inputs(17, B, T, H, dk, dv)
        run = lambda vv: oracle.recur_delta(q, k, vv, beta, S0, scale=1.0)
    else:
        q, k, v, w, S0 = _rwkv_inputs(17, B, T, H, dk, dv)
        run = lambda vv: oracle.recur_rwkv7(q, k, vv, w, S0)
    o1, S1 = run(v)
    v2 = v.copy()
    v2[:, :, 1] += 1.0
    o2, S2 = run(v2)
    for h in (0, 2):
        assert np.array_equal(o1[:, :, h], o2[:, :, h]) and np.array_equal(S1[:, h], S2[:, h])
    assert not np.allclose(o1[:, :, 1], o2[:, :, 1])


# ------------------------------------------------------------------ delta
def test_delta_rank1_matches_explicit_form_and_wrong_side_fails():
    """Rank-1 form == explicit (I - b k k^T) S + b k v^T with dk == dv (fp64);
    the wrong-side products S (I - b k k^T) + b k v^T and the S k (instead of
    S^T k) correction both differ by far more than the tolerance."""
    B, T, H, dk = 1, 30, 2, 6
    q, k, v, beta, S0 = _delta_inputs(20, B, T, H, dk, dk)
    o, S = oracle.recur_delta(q, k, v, beta, S0, scale=1.0)
    for h in range(H):
        M = S0[0, h].copy()
        Mw1 = S0[0, h].copy()
        Mw2 = S0[0, h].copy()
        I = np.eye(dk)
        for t in range(T):
            kk, vv, bt = k[0, t, h].astype(np.float64), v[0, t, h].astype(np.float64), float(beta[0, t, h])
            M = (I - bt * _outer(kk, kk)) @ M + bt * _outer(kk, vv)
            Mw1 = Mw1 @ (I - bt * _outer(kk, kk)) + bt * _outer(kk, vv)
            Mw2 = Mw2 + _outer(kk, (vv - Mw2 @ kk) * bt)
            assert _nrel(o[0, t, h], M.T @ q[0, t, h].astype(np.float64)) < 1e-12
        assert _nrel(S[0, h], M) < 1e-12
        assert _nrel(Mw1, M) > 1e-3
        assert _nrel(Mw2, M) > 1e-3


def test_delta_bruteforce_unrolled():
    """T <= 6: S_T = prod(I - b_t k_t k_t^T) S0 + sum_j prod_{t>j}(...) b_j k_j v_j^T."""
    B, T, H, dk, dv = 1, 6, 1, 5, 3
    q, k, v, beta, S0 = _delta_inputs(21, B, T, H, dk, dv)
    _, S = oracle.recur_delta(q, k, v, beta, S0, scale=1.0)
    A = [np.eye(dk) - float(beta[0, t, 0]) * _outer(k[0, t, 0], k[0, t, 0])
         for t in range(T)]
    P = np.eye(dk)
    for t in range(T):
        P = A[t] @ P
    ref = P @ S0[0, 0]
    for j in range(T):
        Pj = np.eye(dk)
        for t in range(j + 1, T):
            Pj = A[t] @ Pj
        ref = ref + Pj @ (float(beta[0, j, 0]) * _outer(k[0, j, 0], v[0, j, 0]))
    assert _nrel(S[0, 0], ref) < 1e-12


def _exact_unit_keys(seed, shape):
    """Random keys with exactly unit norm in fp32: four entries of +-1/2."""
    rng = _rng(seed)
    dk = shape[-1]
    k = np.zeros(shape, np.float32)
    flat = k.reshape(-1, dk)
    for r in range(flat.shape[0]):
        idx = rng.choice(dk, 4, replace=False)
        flat[r, idx] = rng.choice([-0.5, 0.5], 4)
    return k


def test_delta_retrieval_identities():
    """With q = k: beta = 1 and unit k give S_t^T k_t = v_t; in general
    S_t^T k_t = (1 - beta_t |k_t|^2) S_{t-1}^T k_t + beta_t |k_t|^2 v_t."""
    B, T, H, dk, dv = 1, 20, 2, 8, 6
    _, k, v, beta, S0 = _delta_inputs(22, B, T, H, dk, dv)
    ku = _exact_unit_keys(23, (B, T, H, dk))
    o, _ = oracle.recur_delta(ku, ku, v, np.ones_like(beta), S0, scale=1.0)
    assert np.max(np.abs(o - v)) < 1e-12
    # general one-step identity, t = 0, from the known S0
    o, _ = oracle.recur_delta(k, k, v, beta, S0, scale=1.0)
    for h in range(H):
        kk = k[0, 0, h].astype(np.float64)
        n2, b0 = float(kk @ kk), float(beta[0, 0, h])
        ref = (1 - b0 * n2) * (S0[0, h].T @ kk) + b0 * n2 * v[0, 0, h].astype(np.float64)
        assert np.max(np.abs(o[0, 0, h] - ref)) < 1e-12


# ------------------------------------------------------------------ rwkv7
def test_rwkv7_bruteforce_unrolled():
    """T <= 6: S_T = S0 prod_t M_t + sum_j v_j k_j^T prod_{t>j} M_t with
    M_t = diag(w_t) - k_t k_t^T (the removal uses the state before decay),
    and o_t = S_t q_t at every t."""
    B, T, H, dk, dv = 1, 6, 2, 5, 4
    q, k, v, w, S0 = _rwkv_inputs(30, B, T, H, dk, dv)
    o, S = oracle.recur_rwkv7(q, k, v, w, S0)
    for h in range(H):
        M = [np.diag(w[0, t, h].astype(np.float64)) - _outer(k[0, t, h], k[0, t, h])
             for t in range(T)]
        for tt in range(1, T + 1):
            ref = S0[0, h].copy()
            for t in range(tt):
                ref = ref @ M[t]
            for j in range(tt):
                P = _outer(v[0, j, h], k[0, j, h])
                for t in range(j + 1, tt):
                    P = P @ M[t]
                ref = ref + P
            assert _nrel(o[0, tt - 1, h], ref @ q[0, tt - 1, h].astype(np.float64)) < 1e-12
        assert _nrel(S[0, h], ref) < 1e-12


def test_rwkv7_removal_uses_state_before_decay():
    """Forming the removal term from the decayed state gives a different
    answer, so the brute-force pin distinguishes the two readings."""
    B, T, H, dk, dv = 1, 8, 1, 6, 6
    q, k, v, w, S0 = _rwkv_inputs(31, B, T, H, dk, dv)
    _, S = oracle.recur_rwkv7(q, k, v, w, S0)
    M = S0[0, 0].copy()
    for t in range(T):
        kk, ww, vv = k[0, t, 0].astype(np.float64), w[0, t, 0].astype(np.float64), v[0, t, 0].astype(np.float64)
        Md = M * ww[None, :]
        M = Md - _outer(Md @ kk, kk) + _outer(vv, kk)
    assert _nrel(S[0, 0], M) > 1e-3


def test_rwkv7_no_decay_unit_key_retrieves_value():
    """w = 1 and |k| = 1: S_t k_t = v_t, so with q = k the readout is v_t."""
    B, T, H, dk, dv = 1, 15, 2, 8, 8
    _, _, v, _, S0 = _rwkv_inputs(32, B, T, H, dk, dv)
    k = _exact_unit_keys(33, (B, T, H, dk))
    w = np.ones((B, T, H, dk), np.float32)
    o, _ = oracle.recur_rwkv7(k, k, v, w, S0)
    assert np.max(np.abs(o - v)) < 1e-12


# ------------------------------------------------------------------ common
@pytest.mark.parametrize("fn", ["diag", "diag_head", "delta", "rwkv7"])
@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_matrix_segment_split_bit_exact(fn, prec):
    """Two segments with the state carried equal the full run bit for bit
    ("SunnyNet 工程化实录" §4)."""
    B, T, H, dk, dv, sp = 2, 21, 2, 6, 5, 8
    cast = (lambda x: x) if prec == "f64" else (lambda x: x.astype(np.float32))
    if fn.startswith("diag"):
        per_key = fn == "diag"
        q, k, v, d, S0 = _diag_inputs(40, B, T, H, H, dk, dv, per_key=per_key)
        run = lambda sl, s: oracle.recur_diag(*(np.ascontiguousarray(x[:, sl]) for x in (q, k, v, d)), s,
                                              H=H, G=H, decay_kind=0 if per_key else 1, scale=0.7, prec=prec)
    elif fn == "delta":
        q, k, v, beta, S0 = _delta_inputs(41, B, T, H, dk, dv)
        run = lambda sl, s: oracle.recur_delta(*(np.ascontiguousarray(x[:, sl]) for x in (q, k, v, beta)), s,
                                               scale=0.7, prec=prec)
    else:
        q, k, v, w, S0 = _rwkv_inputs(42, B, T, H, dk, dv)
        run = lambda sl, s: oracle.recur_rwkv7(*(np.ascontiguousarray(x[:, sl]) for x in (q, k, v, w)), s,
                                               prec=prec)
    S0 = cast(S0)
    of, Sf = run(slice(None), S0)
    o1, S1 = run(slice(0, sp), S0)
    o2, S2 = run(slice(sp, None), S1)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), of)
    assert np.array_equal(S2, Sf)


@pytest.mark.parametrize("fn", ["gla", "mamba2", "delta", "rwkv7"])
def test_fp32_oracle_error_vs_fp64(fn):
    """The fp32 oracle's normwise error against fp64 stays well under the 1e-4
    parity bound at workload-shaped inputs ("SunnyNet 工程化实录" §9.3)."""
    import synth
    if fn == "gla":
        x = synth.gla_inputs(1, 256, 2, 64, 64)
        args = [x[n].numpy() for n in ("q", "k", "v", "d")]
        f = lambda p: oracle.recur_diag(*args, H=2, G=2, decay_kind=0, scale=x["scale"], prec=p)
    elif fn == "mamba2":
        x = synth.mamba2_inputs(1, 256, 4, 1, 64, 32)
        args = [x[n].numpy() for n in ("q", "k", "v", "d")]
        f = lambda p: oracle.recur_diag(*args, H=4, G=1, decay_kind=1, scale=1.0, prec=p)
    elif fn == "delta":
        x = synth.deltanet_inputs(1, 256, 2, 64, 64)
        args = [x[n].numpy() for n in ("q", "k", "v", "beta")]
        f = lambda p: oracle.recur_delta(*args, scale=1.0, prec=p)
    else:
        x = synth.rwkv7_inputs(1, 256, 2, 64, 64)
        args = [x[n].numpy() for n in ("q", "k", "v", "w")]
        f = lambda p: oracle.recur_rwkv7(*args, prec=p)
    o64, S64 = f("f64")
    o32, S32 = f("f32")
    assert _nrel(o32, o64) < 1e-5 and _nrel(S32, S64) < 1e-5


# ------------------------------------------------------------------ gated matrix state
def _gated_inputs(seed, B, T, H, dk, dv, per_key=True):
    rng = _rng(seed)
    q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    p = _sig(rng.standard_normal((B, T, H, dk) if per_key else (B, T, H)) + 1.0)
    S0 = rng.standard_normal((B, H, dk, dv)) * 3
    return q, k, v, p, S0


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_gated_hand_fixture(prec):
    g = _golden.load("diag_gated_dyadic.txt")
    B, T, H, G, dk, dv = g["shape"]
    o, S = oracle.recur_diag(_golden.f32(g["q"], (B, T, G, dk)), _golden.f32(g["k"], (B, T, G, dk)),
                             _golden.f32(g["v"], (B, T, H, dv)), _golden.f32(g["d"], (B, T, H, dk)),
                             np.asarray(g["S0"]).reshape(B, H, dk, dv), H=H, G=G,
                             decay_kind=int(g["decay_kind"][0]), scale=1.0, prec=prec)
    assert np.array_equal(o, np.asarray(g["o"]).reshape(B, T, H, dv))
    assert np.array_equal(S, np.asarray(g["S"]).reshape(B, H, dk, dv))


@pytest.mark.parametrize("per_key", [True, False])
def test_gated_state_contracts_to_constant_injection(per_key):
    """Constant k, v: S_t - k v^T = diag(prod p) (S0 - k v^T) (convex
    combination with a fixed point, "我拿同一份权重…" §8: S stays bounded)."""
    B, T, H, dk, dv = 1, 60, 2, 6, 4
    q, k, v, p, S0 = _gated_inputs(50, B, T, H, dk, dv, per_key)
    k[:] = k[:, :1]
    v[:] = v[:, :1]
    kind = oracle.DECAY_PER_KEY_GATED if per_key else oracle.DECAY_PER_HEAD_GATED
    _, S = oracle.recur_diag(q, k, v, p, S0, H=H, G=H, decay_kind=kind, scale=1.0)
    for h in range(H):
        fixed = _outer(k[0, 0, h], v[0, 0, h])
        pr = np.prod(p[0, :, h].astype(np.float64), axis=0)
        P = pr[:, None] if per_key else pr
        assert np.max(np.abs(S[0, h] - (fixed + P * (S0[0, h] - fixed)))) < 1e-12


def test_gated_state_stays_in_convex_hull():
    B, T, H, dk, dv = 1, 200, 1, 5, 3
    q, k, v, p, S0 = _gated_inputs(51, B, T, H, dk, dv)
    _, S = oracle.recur_diag(q, k, v, p, S0, H=H, G=H, decay_kind=oracle.DECAY_PER_KEY_GATED, scale=1.0)
    inj = k[0, :, 0, :, None].astype(np.float64) * v[0, :, 0, None, :]
    lo = np.minimum(inj.min(axis=0), S0[0, 0])
    hi = np.maximum(inj.max(axis=0), S0[0, 0])
    assert np.all(S[0, 0] >= lo - 1e-12) and np.all(S[0, 0] <= hi + 1e-12)


def test_gated_bruteforce_unrolled():
    """T <= 6: S_T = (prod D_t) S0 + sum_j (prod_{t>j} D_t) diag(1 - p_j) k_j v_j^T."""
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    q, k, v, p, S0 = _gated_inputs(52, B, T, H, dk, dv)
    _, S = oracle.recur_diag(q, k, v, p, S0, H=H, G=H, decay_kind=oracle.DECAY_PER_KEY_GATED, scale=1.0)
    for h in range(H):
        D = [np.diag(p[0, t, h].astype(np.float64)) for t in range(T)]
        acc = np.eye(dk)
        for t in range(T):
            acc = D[t] @ acc
        ref = acc @ S0[0, h]
        for j in range(T):
            P = np.eye(dk)
            for t in range(j + 1, T):
                P = D[t] @ P
            ref = ref + P @ np.diag(1.0 - p[0, j, h].astype(np.float64)) @ _outer(k[0, j, h], v[0, j, h])
        assert _nrel(S[0, h], ref) < 1e-13


def test_gated_f32_decomposes_into_fma_scans():
    """Each entry of the fp32 gated state is the FMA-form scan with a = p_i and
    b = fl(fl(fl(1 - p_i) k_i) v_j), bit for bit."""
    B, T, H, dk, dv = 1, 40, 1, 6, 4
    q, k, v, p, S0 = _gated_inputs(53, B, T, H, dk, dv)
    S0 = S0.astype(np.float32)
    _, S = oracle.recur_diag(q, k, v, p, S0, H=H, G=H, decay_kind=oracle.DECAY_PER_KEY_GATED, scale=1.0,
                             prec="f32")
    kg = ((np.float32(1) - p[0, :, 0]) * k[0, :, 0]).astype(np.float32)
    bb = (kg[:, :, None] * v[0, :, 0, None, :]).astype(np.float32)
    a = np.repeat(p[0, :, 0, :, None], dv, axis=2)
    _, sf = oracle.scan_fma(np.ascontiguousarray(a.reshape(1, T, dk * dv)),
                            np.ascontiguousarray(bb.reshape(1, T, dk * dv)), S0[0, 0].reshape(1, dk * dv),
                            prec="f32")
    assert np.array_equal(sf.reshape(dk, dv).view(np.uint32), S[0, 0].view(np.uint32))
