"""Pins of the oracle's gated RMS norm (CPU only): mathematical properties
that a mistake in the gate, the mean, the grouping or the weight breaks."""
import math

import numpy as np

import oracle


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_normalised_groups_have_unit_rms():
    """eps = 0, weight = 1: every group of the output has mean square 1."""
    y, z = rand((3, 5, 48), 1), rand((3, 5, 48), 2)
    out = oracle.gated_rmsnorm(y, z, np.ones(48), 0.0, 16)
    ms = np.mean(out.reshape(3, 5, 3, 16) ** 2, axis=-1)
    assert np.allclose(ms, 1.0, atol=1e-13)


def test_scale_invariance_and_weight():
    """out(c y) = out(y) for c > 0 when eps = 0; the weight multiplies channels."""
    y, z, w = rand((4, 32), 3), rand((4, 32), 4), rand(32, 5)
    a = oracle.gated_rmsnorm(y, z, w, 0.0, 8)
    b = oracle.gated_rmsnorm(7.5 * y, z, w, 0.0, 8)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
    c = oracle.gated_rmsnorm(y, z, np.ones(32), 0.0, 8)
    assert np.allclose(a, c * w, rtol=1e-13, atol=1e-13)


def test_gate_is_silu():
    """Large z: silu(z) = z to double precision, so the gate is y z; and
    silu(z) - silu(-z) = z (read through two one-channel groups, where the
    norm divides by |g|: out = sign(g))."""
    y = rand((2, 6), 6)
    z = np.full((2, 6), 40.0)
    got = oracle.gated_rmsnorm(y, z, np.ones(6), 0.0, 6)
    g = y * 40.0
    ref = g / np.sqrt(np.mean(g * g, axis=-1, keepdims=True))
    assert np.allclose(got, ref, rtol=1e-14)
    # silu(0.7) - silu(-0.7) = 0.7: with y = 1 and group size 2 over [z, -z]
    s = lambda v: v / (1.0 + math.exp(-v))
    zz = np.array([[0.7, -0.7]])
    out = oracle.gated_rmsnorm(np.ones((1, 2)), zz, np.ones(2), 0.0, 2)
    a, b = s(0.7), s(-0.7)
    assert abs((a - b) - 0.7) < 1e-15
    rms = math.sqrt((a * a + b * b) / 2)
    assert np.allclose(out, [[a / rms, b / rms]], rtol=1e-14)


def test_groups_are_independent():
    """Changing one group's inputs leaves the other groups' outputs unchanged."""
    y, z, w = rand((2, 24), 7), rand((2, 24), 8), rand(24, 9)
    a = oracle.gated_rmsnorm(y, z, w, 1e-5, 8)
    y2 = y.copy()
    y2[:, 8:16] *= 3.0
    y2[:, 9] += 1.0
    b = oracle.gated_rmsnorm(y2, z, w, 1e-5, 8)
    assert np.array_equal(a[:, :8], b[:, :8]) and np.array_equal(a[:, 16:], b[:, 16:])
    assert not np.allclose(a[:, 8:16], b[:, 8:16])


def test_eps_bounds_small_groups():
    """An all-zero group stays zero (no division by zero) and eps enters as
    mean square + eps: g = c constant gives c / sqrt(c^2 + eps)."""
    y = np.zeros((1, 8))
    out = oracle.gated_rmsnorm(y, rand((1, 8), 10), np.ones(8), 1e-6, 4)
    assert np.array_equal(out, np.zeros((1, 8)))
    z = np.full((1, 4), 40.0)
    y = np.full((1, 4), 0.5 / 40.0)  # g = 0.5 everywhere
    out = oracle.gated_rmsnorm(y, z, np.ones(4), 0.01, 4)
    assert np.allclose(out, 0.5 / math.sqrt(0.25 + 0.01), rtol=1e-13)
