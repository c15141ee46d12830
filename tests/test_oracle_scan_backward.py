"""Pins of the oracle's reverse (adjoint) scans.

Source: "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时" §2.1
(forward forms) and §8 (the kernels ship forward-scan, reverse-scan and
single-step entries).  The reverse scan is the adjoint of the forward scan;
each check below comes from the mathematics, not from the oracle itself:
hand fixtures, exact rational unrolled sums, the adjoint dot-product identity
against an independent tangent-linear recurrence, and closed-form cases.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _golden


def _rng(seed):
    return np.random.default_rng(seed)


def _sig(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_hand_fixtures(prec):
    g = _golden.load("scan_backward_dyadic.txt")
    sh = (1, 3, 1)
    for form in ("fma", "gated"):
        a = _golden.f32(g[f"{form}_a"], sh)
        rhs = _golden.f32(g[f"{form}_b" if form == "fma" else "gated_u"], sh)
        s0 = np.asarray(g[f"{form}_s0"]).reshape(1, 1)
        fwd = oracle.scan_fma if form == "fma" else oracle.scan_gated
        s, _ = fwd(a, rhs, s0, prec=prec)
        da, dbu, ds0 = oracle.scan_backward(form, a, s, s0, _golden.f32(g[f"{form}_gs"], sh),
                                            _golden.f32(g[f"{form}_gf"], (1, 1)),
                                            u=rhs if form == "gated" else None, prec=prec)
        assert np.array_equal(da.ravel(), g[f"{form}_da"])
        assert np.array_equal(dbu.ravel(), g[f"{form}_db" if form == "fma" else "gated_du"])
        assert np.array_equal(ds0.ravel(), g[f"{form}_ds0"])


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_exact_unrolled_adjoint(form):
    """T <= 7: g_t = sum_{tau >= t} gs_tau prod_{t < r <= tau} a_r
    + gf prod_{t < r < T} a_r, and the input gradients from it, as exact
    rationals over an exact rational forward pass."""
    rng = _rng(1)
    B, T, N = 1, 7, 2
    a = _sig(rng.standard_normal((B, T, N)))
    rhs = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N))
    gs = rng.standard_normal((B, T, N)).astype(np.float32)
    gf = rng.standard_normal((B, N)).astype(np.float32)
    fwd = oracle.scan_fma if form == "fma" else oracle.scan_gated
    s, _ = fwd(a, rhs, s0)
    da, dbu, ds0 = oracle.scan_backward(form, a, s, s0, gs, gf, u=rhs if form == "gated" else None)
    F = lambda x: Fraction(float(x))
    for n in range(N):
        A = [F(a[0, t, n]) for t in range(T)]
        R = [F(rhs[0, t, n]) for t in range(T)]
        S = []
        prev = F(s0[0, n])
        for t in range(T):
            prev = A[t] * prev + (R[t] if form == "fma" else (1 - A[t]) * R[t])
            S.append(prev)
        for t in range(T):
            g = Fraction(0)
            for tau in range(t, T):
                P = Fraction(1)
                for r in range(t + 1, tau + 1):
                    P *= A[r]
                g += F(gs[0, tau, n]) * P
            P = Fraction(1)
            for r in range(t + 1, T):
                P *= A[r]
            g += F(gf[0, n]) * P
            sprev = S[t - 1] if t > 0 else F(s0[0, n])
            if form == "fma":
                ea, eb = g * sprev, g
            else:
                ea, eb = g * (sprev - R[t]), g * (1 - A[t])
            assert abs(da[0, t, n] - float(ea)) <= 1e-13 * max(1.0, abs(float(ea)))
            assert abs(dbu[0, t, n] - float(eb)) <= 1e-13 * max(1.0, abs(float(eb)))
            if t == 0:
                assert abs(ds0[0, n] - float(A[0] * g)) <= 1e-13 * max(1.0, abs(float(A[0] * g)))


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_adjoint_dot_product_identity(form):
    """<gs, ds> + <gf, ds_final> == <da, δa> + <db|du, δb|δu> + <ds0, δs0>
    for random directions, where ds is the tangent-linear forward
    δs_t = a_t δs_{t-1} + δa_t s_{t-1} + δb_t (gated: + δa_t (s_{t-1} - u_t)
    ... written out from the forward step, independent of the reverse scan)."""
    rng = _rng(2)
    B, T, N = 2, 300, 5
    a = _sig(rng.standard_normal((B, T, N)) + 1.0)
    rhs = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N))
    gs = rng.standard_normal((B, T, N)).astype(np.float32)
    gf = rng.standard_normal((B, N)).astype(np.float32)
    fwd = oracle.scan_fma if form == "fma" else oracle.scan_gated
    s, sf = fwd(a, rhs, s0)
    da, dbu, ds0 = oracle.scan_backward(form, a, s, s0, gs, gf, u=rhs if form == "gated" else None)
    A = a.astype(np.float64)
    Rr = rhs.astype(np.float64)
    ea, er, e0 = rng.standard_normal((B, T, N)), rng.standard_normal((B, T, N)), rng.standard_normal((B, N))
    ds = np.empty((B, T, N))
    prev_ds = e0.copy()
    prev_s = s0.copy()
    for t in range(T):
        if form == "fma":
            cur = A[:, t] * prev_ds + ea[:, t] * prev_s + er[:, t]
        else:
            cur = A[:, t] * prev_ds + ea[:, t] * (prev_s - Rr[:, t]) + (1 - A[:, t]) * er[:, t]
        ds[:, t] = cur
        prev_ds, prev_s = cur, s[:, t]
    lhs = np.sum(gs * ds) + np.sum(gf * ds[:, -1])
    rhs_ = np.sum(da * ea) + np.sum(dbu * er) + np.sum(ds0 * e0)
    assert abs(lhs - rhs_) <= 1e-11 * max(1.0, abs(lhs))


def test_closed_form_special_cases():
    """a = 1: g_t is the suffix sum of gs (plus gf); a = 0: g_t = gs_t."""
    rng = _rng(3)
    B, T, N = 1, 50, 3
    gs = rng.standard_normal((B, T, N)).astype(np.float32)
    gf = rng.standard_normal((B, N)).astype(np.float32)
    b = np.zeros((B, T, N), np.float32)
    ones = np.ones((B, T, N), np.float32)
    s, _ = oracle.scan_fma(ones, b, np.zeros((B, N)))
    _, db, ds0 = oracle.scan_backward("fma", ones, s, None, gs, gf)
    suffix = np.cumsum(gs[:, ::-1].astype(np.float64), axis=1)[:, ::-1] + gf[:, None, :]
    assert np.max(np.abs(db - suffix)) < 1e-12
    assert np.max(np.abs(ds0 - suffix[:, 0])) < 1e-12
    zeros = np.zeros((B, T, N), np.float32)
    s, _ = oracle.scan_fma(zeros, b)
    _, db, ds0 = oracle.scan_backward("fma", zeros, s, None, gs, gf)
    expect = gs.astype(np.float64).copy()
    expect[:, -1] += gf
    assert np.array_equal(db, expect) and np.all(ds0 == 0)


@pytest.mark.parametrize("form", ["fma", "gated"])
def test_fp32_reverse_error_vs_fp64(form):
    rng = _rng(4)
    B, T, N = 2, 2048, 16
    a = _sig(rng.standard_normal((B, T, N)) + 1.5)
    rhs = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N)).astype(np.float32)
    gs = rng.standard_normal((B, T, N)).astype(np.float32)
    fwd = oracle.scan_fma if form == "fma" else oracle.scan_gated
    s32, _ = fwd(a, rhs, s0, prec="f32")
    u = rhs if form == "gated" else None
    r64 = oracle.scan_backward(form, a, s32.astype(np.float64), s0.astype(np.float64), gs, None, u=u)
    r32 = oracle.scan_backward(form, a, s32, s0, gs, None, u=u, prec="f32")
    for x32, x64 in zip(r32, r64):
        assert np.max(np.abs(x32 - x64)) / np.max(np.abs(x64)) < 2e-6
