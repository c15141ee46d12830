"""Pins of the oracle's readout epilogues against what the mathematics fixes.

GLA readout y = RMSNorm(o) * w * silu(g), normalised first and gated after
("SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时" §4.3); the
Mamba-2 skip connection y = o + D_h x (same page, §4.1, readout of each head).
"""
import numpy as np
import pytest

import oracle
from tests import _golden


def _rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def test_norm_gate_hand_fixture():
    f = _golden.load("readout_norm_gate.txt")
    shape = f["shape"]
    y = oracle.readout_norm_gate(_golden.f32(f["o"], shape), _golden.f32(f["g"], shape),
                                 _golden.f32(f["w"], shape[-1:]), eps=0.0)
    np.testing.assert_allclose(y, np.asarray(f["y"]).reshape(shape), rtol=1e-15, atol=1e-14)


def test_norm_gate_matches_an_independent_formulation():
    """rms = ||o||_2 / sqrt(dv) and silu(g) = g (1 + tanh(g / 2)) / 2: other
    formulas for the same functions."""
    o, g, w = _rand((5, 3, 64), 1), _rand((5, 3, 64), 2, 3.0), _rand((64,), 3)
    eps = 1e-3
    o64, g64 = o.astype(np.float64), g.astype(np.float64)
    rms = np.sqrt(np.linalg.norm(o64, axis=-1, keepdims=True) ** 2 / 64 + eps)
    ref = o64 / rms * w.astype(np.float64) * (g64 * 0.5 * (1.0 + np.tanh(g64 / 2)))
    np.testing.assert_allclose(oracle.readout_norm_gate(o, g, w, eps=eps), ref, rtol=1e-12, atol=1e-13)


def test_norm_gate_scale_invariance():
    """RMSNorm(c o) with eps c^2 equals RMSNorm(o) with eps, for c > 0."""
    o, g, w = _rand((4, 128), 4), _rand((4, 128), 5), _rand((128,), 6)
    c = np.float32(8.0)                      # a power of two keeps c * o exact in fp32
    y1 = oracle.readout_norm_gate(o, g, w, eps=1e-4)
    y2 = oracle.readout_norm_gate(o * c, g, w, eps=1e-4 * 64.0)
    np.testing.assert_allclose(y2, y1, rtol=1e-13, atol=1e-15)


def test_norm_gate_rows_have_unit_rms_before_weight_and_gate():
    """With eps = 0, y / (w silu(g)) has root mean square 1 in every row: the
    normalisation runs over the value channels of one (b, t, h)."""
    o, g, w = _rand((6, 7, 64), 7), _rand((6, 7, 64), 8) + 3.0, _rand((64,), 9) + 2.0
    y = oracle.readout_norm_gate(o, g, w, eps=0.0)
    g64 = g.astype(np.float64)
    z = y / (w.astype(np.float64) * g64 / (1 + np.exp(-g64)))
    np.testing.assert_allclose(np.sqrt(np.mean(z * z, axis=-1)), 1.0, rtol=1e-12)


def test_norm_gate_normalises_before_gating():
    """The other order, RMSNorm(o * silu(g)) * w, gives a different result."""
    o, g = _rand((3, 64), 10), _rand((3, 64), 11)
    y = oracle.readout_norm_gate(o, g, None, eps=0.0)
    s = o * (g / (1 + np.exp(-g)))
    other = oracle.readout_norm_gate(s.astype(np.float32), np.full_like(g, 40.0), None, eps=0.0) / 40.0
    assert np.max(np.abs(y - other)) > 1e-2


def test_norm_gate_zero_row_with_eps_and_zero_gate():
    o, g = np.zeros((2, 64), np.float32), _rand((2, 64), 12)
    assert np.all(oracle.readout_norm_gate(o, g, None, eps=1e-6) == 0.0)
    o2 = _rand((2, 64), 13)
    assert np.all(oracle.readout_norm_gate(o2, np.zeros_like(o2), None, eps=1e-6) == 0.0)


def test_dskip_hand_fixture():
    f = _golden.load("readout_dskip.txt")
    shape = f["shape"]
    y = oracle.readout_dskip(_golden.f32(f["o"], shape), _golden.f32(f["x"], shape),
                             _golden.f32(f["D"], (shape[2],)))
    assert np.array_equal(y, np.asarray(f["y"]).reshape(shape))


def test_dskip_head_mapping_and_zero_skip():
    o, x = _rand((2, 5, 3, 64), 14), _rand((2, 5, 3, 64), 15)
    D = np.array([0.5, -1.25, 2.0], np.float32)
    y = oracle.readout_dskip(o, x, D)
    for h in range(3):
        np.testing.assert_allclose(y[:, :, h] - o[:, :, h], D[h] * x[:, :, h].astype(np.float64), rtol=1e-15,
                                   atol=1e-15)
    assert np.array_equal(oracle.readout_dskip(o, x, np.zeros(3, np.float32)), o.astype(np.float64))
