"""Pins of the oracle's RMSNorm and NeoX RoPE (CPU only)."""
import math

import numpy as np


def test_rmsnorm_all_ones_gives_the_weight(orc):
    # dflash/forward.rs, smoke_input_norm_and_q_proj: at an all-ones input the
    # normalised value equals the weight (up to the eps term).
    w = np.linspace(0.5, 1.5, 256).astype(np.float32)
    y = orc.rmsnorm(np.ones(256), w, eps=1e-6)
    assert np.max(np.abs(y - w.astype(np.float64))) <= 1e-6


def test_rmsnorm_unit_weight_has_unit_rms(orc):
    x = np.random.default_rng(0).normal(size=128) * 7.0
    y = orc.rmsnorm(x, None, eps=0.0)
    assert abs(np.mean(y * y) - 1.0) <= 1e-14


def test_rmsnorm_is_scale_invariant_without_eps(orc):
    x = np.random.default_rng(1).normal(size=64)
    assert np.max(np.abs(orc.rmsnorm(x, None, 0.0) - orc.rmsnorm(1e3 * x, None, 0.0))) <= 1e-13


def test_rmsnorm_eps_sits_under_the_root_next_to_the_mean(orc):
    # x = 1e-3 everywhere, eps = 1e-6: mean(x^2) = 1e-6, so y = 1e-3 / sqrt(2e-6).
    y = orc.rmsnorm(np.full(32, 1e-3), None, eps=1e-6)
    assert np.allclose(y, 1e-3 / math.sqrt(2e-6), rtol=1e-14, atol=0)


def test_rope_hand_computed_angles(orc):
    # head_dim 4, theta 1e4, position 1: pair (0, 2) turns by 1 rad and pair (1, 3)
    # by theta^(-2/4) = 0.01 rad (NeoX pairing i <-> i + hd/2, counter-clockwise).
    u = orc.rope_neox([1.0, 2.0, 3.0, 4.0], pos=1, theta=1e4)
    c1, s1, c2, s2 = math.cos(1.0), math.sin(1.0), math.cos(0.01), math.sin(0.01)
    expect = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 1 * s1 + 3 * c1, 2 * s2 + 4 * c2]
    assert np.allclose(u, expect, rtol=0, atol=1e-15)


def test_rope_power_of_two_frequencies(orc):
    # theta = 16, head_dim 8: inverse frequencies 16^(-2i/8) = 2^-i exactly.
    for i in range(4):
        e = np.zeros(8)
        e[i] = 1.0
        u = orc.rope_neox(e, pos=3, theta=16.0)
        phi = 3 * 2.0 ** -i
        assert abs(u[i] - math.cos(phi)) < 1e-15 and abs(u[i + 4] - math.sin(phi)) < 1e-15
        assert np.count_nonzero(np.abs(u) > 1e-15) <= 2


def test_rope_position_zero_is_identity(orc):
    u = np.random.default_rng(2).normal(size=128)
    assert np.array_equal(orc.rope_neox(u, 0, 1e6), u)


def test_rope_preserves_pair_norms_and_composes(orc):
    rng = np.random.default_rng(3)
    u = rng.normal(size=128)
    a = orc.rope_neox(u, 1000, 1e6)
    n0 = u[:64] ** 2 + u[64:] ** 2
    n1 = a[:64] ** 2 + a[64:] ** 2
    assert np.max(np.abs(n1 - n0) / n0) <= 1e-13
    b = orc.rope_neox(a, 234, 1e6)
    c = orc.rope_neox(u, 1234, 1e6)
    assert np.max(np.abs(b - c)) <= 1e-11
    back = orc.rope_neox(a, -1000, 1e6)
    assert np.max(np.abs(back - u)) <= 1e-11


def test_rope_scores_depend_on_relative_position_only(orc):
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=64), rng.normal(size=64)
    s1 = orc.rope_neox(q, 500, 1e4) @ orc.rope_neox(k, 480, 1e4)
    s2 = orc.rope_neox(q, 9000, 1e4) @ orc.rope_neox(k, 8980, 1e4)
    assert abs(s1 - s2) <= 1e-10
