"""Pins of the CPU oracle's scans against what the pages and mathematics fix.

Source: "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
§2.1 (FMA and gated forms), §4 (segment-split continuation is bit-exact),
§9.3 (fp32 scan error is small).  Nothing here compares the oracle with
itself: each check is a closed form, an invariant, exact rational brute force
or a hand-derived fixture.
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


# ---------------------------------------------------------------- fixtures
@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_fma_hand_fixture(prec):
    g = _golden.load("scan_fma_dyadic.txt")
    B, T, N = g["shape"]
    a, b = _golden.f32(g["a"], (B, T, N)), _golden.f32(g["b"], (B, T, N))
    s_out, s_fin = oracle.scan_fma(a, b, np.asarray(g["s0"]).reshape(B, N), prec=prec)
    assert np.array_equal(s_out, np.asarray(g["s_out"]).reshape(B, T, N))
    assert np.array_equal(s_fin, np.asarray(g["s_final"]).reshape(B, N))


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_gated_hand_fixture(prec):
    g = _golden.load("scan_gated_dyadic.txt")
    B, T, N = g["shape"]
    a, u = _golden.f32(g["a"], (B, T, N)), _golden.f32(g["u"], (B, T, N))
    s_out, s_fin = oracle.scan_gated(a, u, np.asarray(g["s0"]).reshape(B, N), prec=prec)
    assert np.array_equal(s_out, np.asarray(g["s_out"]).reshape(B, T, N))
    assert np.array_equal(s_fin, np.asarray(g["s_final"]).reshape(B, N))


# ---------------------------------------------------------------- closed forms
def test_fma_constant_coefficients_closed_form():
    """Constant a and b: s_T = a^T s0 + b (1 - a^T) / (1 - a), exact rationals."""
    B, T, N = 1, 300, 4
    a_vals = np.array([0.8, 0.5, 0.999, 0.1], np.float32)
    b_vals = np.array([1.0, -2.5, 0.01, 3.0], np.float32)
    s0 = np.array([[1.5, 0.0, -4.0, 2.0]])
    a = np.broadcast_to(a_vals, (B, T, N)).copy()
    b = np.broadcast_to(b_vals, (B, T, N)).copy()
    s_out, s_fin = oracle.scan_fma(a, b, s0)
    for n in range(N):
        A, Bv, S0 = Fraction(float(a_vals[n])), Fraction(float(b_vals[n])), Fraction(float(s0[0, n]))
        for t in (0, 1, 7, 63, T - 1):
            p = A ** (t + 1)
            exact = p * S0 + Bv * (1 - p) / (1 - A)
            got = Fraction(float(s_out[0, t, n]))
            assert abs(got - exact) <= Fraction(1, 10 ** 13) * max(1, abs(exact))
    assert np.array_equal(s_fin, s_out[:, -1, :])


def test_fma_constant_a_long_sequence():
    """Constant a, arbitrary b: s_t = a^{t+1} s0 + sum_j a^{t-j} b_j.  Checked at
    T = 8192 in extended precision (numpy longdouble) to 1e-12 relative."""
    T = 8192
    rng = _rng(1)
    a_val = np.float32(0.82)
    b = rng.standard_normal((1, T, 1)).astype(np.float32)
    a = np.full((1, T, 1), a_val, np.float32)
    s0 = np.array([[0.7]])
    s_out, _ = oracle.scan_fma(a, b, s0)
    al = np.longdouble(a_val)
    ref = np.longdouble(0.7)
    refs = np.empty(T, np.longdouble)
    for t in range(T):                      # Horner form of the closed-form sum
        ref = al * ref + np.longdouble(b[0, t, 0])
        refs[t] = ref
    scale = np.max(np.abs(refs))
    assert np.max(np.abs(s_out[0, :, 0] - refs)) / scale < 1e-12


def test_fma_unrolled_bruteforce_exact():
    """T <= 8: s_t = (prod_{r<=t} a_r) s0 + sum_{j<=t} (prod_{j<r<=t} a_r) b_j,
    evaluated as exact rationals."""
    rng = _rng(2)
    B, T, N = 2, 8, 3
    a = _sig(rng.standard_normal((B, T, N)))
    b = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N))
    s64, _ = oracle.scan_fma(a, b, s0)
    s32, _ = oracle.scan_fma(a, b, s0.astype(np.float32), prec="f32")
    for bi in range(B):
        for n in range(N):
            for t in range(T):
                P = Fraction(1)
                for r in range(t + 1):
                    P *= Fraction(float(a[bi, r, n]))
                exact = P * Fraction(float(s0[bi, n]))
                for j in range(t + 1):
                    Pj = Fraction(1)
                    for r in range(j + 1, t + 1):
                        Pj *= Fraction(float(a[bi, r, n]))
                    exact += Pj * Fraction(float(b[bi, j, n]))
                e = float(exact)
                assert abs(s64[bi, t, n] - e) <= 1e-14 * max(1.0, abs(e))
                assert abs(float(s32[bi, t, n]) - e) <= 4e-6 * max(1.0, abs(e))


def test_gated_constant_u_contracts_to_u():
    """Constant u: s_t - u = (prod a)(s0 - u), so s -> u."""
    rng = _rng(3)
    B, T, N = 1, 400, 5
    a = _sig(rng.standard_normal((B, T, N)))
    u_val = rng.standard_normal(N).astype(np.float32)
    u = np.broadcast_to(u_val, (B, T, N)).copy()
    s0 = np.array([[5.0, -3.0, 0.0, 10.0, -0.5]])
    s_out, _ = oracle.scan_gated(a, u, s0)
    P = np.cumprod(a[0].astype(np.float64), axis=0)
    expect = u_val[None, :] + P * (s0[0] - u_val)[None, :]
    assert np.max(np.abs(s_out[0] - expect)) < 1e-13
    assert np.max(np.abs(s_out[0, -1] - u_val)) < 1e-6


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_gated_convex_hull(prec):
    """Every gated state is a convex combination of s0 and u_0..u_t, so it stays
    inside their running [min, max] (to a few ulps of rounding)."""
    rng = _rng(4)
    B, T, N = 2, 500, 16
    a = _sig(rng.standard_normal((B, T, N)))
    u = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N)) * 3
    s_out, _ = oracle.scan_gated(a, u, s0, prec=prec)
    lo = np.minimum(np.minimum.accumulate(u, axis=1), s0[:, None, :].astype(np.float32))
    hi = np.maximum(np.maximum.accumulate(u, axis=1), s0[:, None, :].astype(np.float32))
    eps = 4 * np.finfo(np.float32 if prec == "f32" else np.float64).eps * 4
    assert np.all(s_out >= lo - eps) and np.all(s_out <= hi + eps)


def test_gated_f32_order_is_fma_of_rounded_injection():
    """The fp32 gated scan equals the fp32 FMA scan fed b = fl(fl(1 - a) * u):
    the canonical single-precision order forms the injection first."""
    rng = _rng(5)
    B, T, N = 2, 64, 33
    a = _sig(rng.standard_normal((B, T, N)))
    u = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N)).astype(np.float32)
    b = ((np.float32(1.0) - a) * u).astype(np.float32)
    g, gf = oracle.scan_gated(a, u, s0, prec="f32")
    f, ff = oracle.scan_fma(a, b, s0, prec="f32")
    assert np.array_equal(g.view(np.uint32), f.view(np.uint32))
    assert np.array_equal(gf.view(np.uint32), ff.view(np.uint32))


def test_fma_f32_is_single_rounding_per_step():
    """One fp32 step equals a*s+b rounded once to the nearest float (the
    fused multiply-add of the canonical order), checked with exact rationals."""
    rng = _rng(6)
    a = _sig(rng.standard_normal((1, 1, 4096)))
    b = rng.standard_normal((1, 1, 4096)).astype(np.float32)
    s0 = rng.standard_normal((1, 4096)).astype(np.float32)
    s, _ = oracle.scan_fma(a, b, s0, prec="f32")
    exact = [Fraction(float(x)) * Fraction(float(y)) + Fraction(float(z))
             for x, y, z in zip(a.ravel(), s0.ravel(), b.ravel())]
    ref = np.array([float(e) for e in exact]).astype(np.float32)
    # the nearest float to the exact value is among ref and its two neighbours
    for i, e in enumerate(exact):
        c = float(ref[i])
        lo, hi = np.nextafter(np.float32(c), np.float32(-np.inf)), np.nextafter(np.float32(c), np.float32(np.inf))
        best = min((np.float32(c), lo, hi), key=lambda f: abs(Fraction(float(f)) - e))
        assert s[0, 0, i] == best


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("kind", ["fma", "gated"])
@pytest.mark.parametrize("prec", ["f64", "f32"])
@pytest.mark.parametrize("split", [1, 37, 100])
def test_segment_split_bit_exact(kind, prec, split):
    """Running T1 then T2 from the carried state equals the full run bit for
    bit ("SunnyNet 工程化实录" §4: segment continuation gives 0.0 difference)."""
    rng = _rng(7)
    B, T, N = 2, 160, 9
    a = _sig(rng.standard_normal((B, T, N)) + 1.5)
    b = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N)).astype(np.float32 if prec == "f32" else np.float64)
    fn = oracle.scan_fma if kind == "fma" else oracle.scan_gated
    full, ffin = fn(a, b, s0, prec=prec)
    p1, f1 = fn(np.ascontiguousarray(a[:, :split]), np.ascontiguousarray(b[:, :split]), s0, prec=prec)
    p2, f2 = fn(np.ascontiguousarray(a[:, split:]), np.ascontiguousarray(b[:, split:]), f1, prec=prec)
    assert np.array_equal(np.concatenate([p1, p2], axis=1), full)
    assert np.array_equal(f2, ffin)


@pytest.mark.parametrize("kind", ["fma", "gated"])
def test_fp32_error_vs_fp64_small(kind):
    """fp32 accumulated error stays far below the 1e-5 parity bound
    ("SunnyNet 工程化实录" §9.3 reports ~4.7e-7 relative for fp32 scans)."""
    rng = _rng(8)
    B, T, N = 2, 2048, 64
    a = _sig(rng.standard_normal((B, T, N)) + 1.5)
    b = rng.standard_normal((B, T, N)).astype(np.float32)
    s0 = rng.standard_normal((B, N)).astype(np.float32)
    fn = oracle.scan_fma if kind == "fma" else oracle.scan_gated
    r64, _ = fn(a, b, s0.astype(np.float64))
    r32, _ = fn(a, b, s0, prec="f32")
    err = np.max(np.abs(r32 - r64)) / np.max(np.abs(r64))
    assert err < 2e-6


def test_oracle_catches_planted_mistakes():
    """Sanity of the pins themselves: a recurrence with a dropped term or a
    swapped operand fails the exact fixture, so the fixtures can fail."""
    g = _golden.load("scan_fma_dyadic.txt")
    B, T, N = g["shape"]
    a = np.asarray(g["a"]).reshape(B, T, N)
    b = np.asarray(g["b"]).reshape(B, T, N)
    want = np.asarray(g["s_out"]).reshape(B, T, N)
    s0 = np.asarray(g["s0"]).reshape(B, N)

    def run(step):
        s = s0[0].copy()
        out = []
        for t in range(T):
            s = step(a[0, t], s, b[0, t])
            out.append(s.copy())
        return np.array(out)[None]
    assert np.array_equal(run(lambda a_, s, b_: a_ * s + b_), want)
    assert not np.array_equal(run(lambda a_, s, b_: a_ * s), want)           # dropped b
    assert not np.array_equal(run(lambda a_, s, b_: b_ * s + a_), want)      # swapped a, b
    assert not np.array_equal(run(lambda a_, s, b_: (1 - a_) * s + b_), want)
