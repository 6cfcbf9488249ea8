"""Pins of the oracle's RoPE and LayerNorm steps.

RoPE: position 0 is the identity; each pair keeps its norm; scores depend
only on relative position; the rotation equals complex multiplication done in
float64 by numpy; NeoX equals GPT-J on a permuted vector.  LayerNorm: with
gamma = 1, beta = 0 the output has mean 0 and variance sigma^2/(sigma^2+eps);
a constant row gives beta exactly; the result agrees with CPU torch's
layer_norm in float64.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

R = 64
HALF = R // 2


def _pairs(style):
    i = np.arange(HALF)
    return (i, i + HALF) if style == oracle.NEOX else (2 * i, 2 * i + 1)


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_position_zero_is_identity(style):
    cos, sin = synth.rope_table(4, R)
    assert np.all(cos[0] == 1.0) and np.all(sin[0] == 0.0)
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((50, 128)) * 10).astype(np.float32)
    y = oracle.rope(x, np.repeat(cos[:1], 50, 0), np.repeat(sin[:1], 50, 0), R, style)
    assert np.array_equal(y.view(np.uint32), x.view(np.uint32))


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_rotation_keeps_pair_norm_and_tail(style):
    rng = np.random.default_rng(2)
    cos, sin = synth.rope_table(262144, R)
    pos = rng.integers(0, 262144, 200)
    x = (rng.standard_normal((200, 128)) * 3).astype(np.float32)
    y = oracle.rope(x, cos[pos], sin[pos], R, style)
    a, b = _pairs(style)
    n0 = x[:, a].astype(np.float64) ** 2 + x[:, b].astype(np.float64) ** 2
    n1 = y[:, a].astype(np.float64) ** 2 + y[:, b].astype(np.float64) ** 2
    assert np.all(np.abs(n1 - n0) <= 1e-6 * n0 + 1e-30)
    assert np.array_equal(y[:, R:], x[:, R:])


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_rotation_is_complex_multiplication(style):
    rng = np.random.default_rng(3)
    cos, sin = synth.rope_table(131072, R)
    pos = rng.integers(0, 131072, 300)
    x = (rng.standard_normal((300, 128)) * 5).astype(np.float32)
    y = oracle.rope(x, cos[pos], sin[pos], R, style)
    a, b = _pairs(style)
    z = (x[:, a].astype(np.float64) + 1j * x[:, b].astype(np.float64)) * (
        cos[pos].astype(np.float64) + 1j * sin[pos].astype(np.float64))
    scale = np.abs(z) + 1e-30
    assert np.all(np.abs(y[:, a] - z.real) <= 4e-7 * scale)
    assert np.all(np.abs(y[:, b] - z.imag) <= 4e-7 * scale)


def test_scores_depend_only_on_relative_position():
    """<R_m q, R_n k> == <R_(m+d) q, R_(n+d) k> (float32 tolerance)."""
    rng = np.random.default_rng(4)
    cos, sin = synth.rope_table(40000, R)
    for style in (oracle.NEOX, oracle.GPTJ):
        q = (rng.standard_normal((64, 128))).astype(np.float32)
        k = (rng.standard_normal((64, 128))).astype(np.float32)
        m = rng.integers(0, 20000, 64)
        n = rng.integers(0, 20000, 64)
        d = rng.integers(0, 19999, 64)
        s0 = np.sum(oracle.rope(q, cos[m], sin[m], R, style).astype(np.float64)
                    * oracle.rope(k, cos[n], sin[n], R, style), axis=1)
        s1 = np.sum(oracle.rope(q, cos[m + d], sin[m + d], R, style).astype(np.float64)
                    * oracle.rope(k, cos[n + d], sin[n + d], R, style), axis=1)
        norm = np.linalg.norm(q, axis=1) * np.linalg.norm(k, axis=1)
        assert np.all(np.abs(s0 - s1) <= 2e-5 * norm)
        # a wrong sign in one term of the rotation would break this:
        flip = oracle.rope(q, cos[m], -sin[m], R, style).astype(np.float64)
        s_flip = np.sum(flip * oracle.rope(k, cos[n], sin[n], R, style), axis=1)
        assert np.max(np.abs(s_flip - s0)) > 1e-2


def test_neox_equals_gptj_on_permuted_vector():
    rng = np.random.default_rng(5)
    cos, sin = synth.rope_table(8192, R)
    pos = rng.integers(0, 8192, 100)
    x = rng.standard_normal((100, 128)).astype(np.float32)
    perm = np.arange(128)
    perm[np.arange(HALF) * 2] = np.arange(HALF)          # GPT-J slot 2i <- NeoX i
    perm[np.arange(HALF) * 2 + 1] = np.arange(HALF) + HALF
    xg = x[:, perm]
    yn = oracle.rope(x, cos[pos], sin[pos], R, oracle.NEOX)
    yg = oracle.rope(xg, cos[pos], sin[pos], R, oracle.GPTJ)
    assert np.array_equal(yg, yn[:, perm])


def test_table_angles_add():
    """cos/sin rows compose: row(m+n) = row(m) * row(n) as unit complex numbers,
    and frequency 0 turns by exactly one radian per position."""
    cos, sin = synth.rope_table(5000, R)
    z = cos.astype(np.float64) + 1j * sin.astype(np.float64)
    rng = np.random.default_rng(6)
    m = rng.integers(0, 2500, 200)
    n = rng.integers(0, 2500, 200)
    assert np.max(np.abs(z[m] * z[n] - z[m + n])) < 1e-6
    assert np.max(np.abs(np.abs(z) - 1)) < 1e-6
    p = np.arange(5000)
    assert np.max(np.abs(z[:, 0] - np.exp(1j * p))) < 1e-6


def test_layernorm_unit_affine_moments():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((300, 128)) * rng.uniform(0.01, 30, (300, 1))
         + rng.uniform(-5, 5, (300, 1))).astype(np.float32)
    eps = 1e-6
    y = oracle.layernorm(x, np.ones(128, np.float32), np.zeros(128, np.float32), eps)
    y64 = y.astype(np.float64)
    var_x = x.astype(np.float64).var(axis=1)
    assert np.all(np.abs(y64.mean(axis=1)) <= 1e-6)
    assert np.all(np.abs(y64.var(axis=1) - var_x / (var_x + eps)) <= 1e-5)


def test_layernorm_constant_row_gives_beta():
    rng = np.random.default_rng(8)
    beta = (rng.standard_normal(128) * 0.1).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    x = np.full((3, 128), 2.5, np.float32)
    x[1] = 0.0
    x[2] = -7.0
    y = oracle.layernorm(x, gamma, beta, 1e-6)
    assert np.array_equal(y, np.broadcast_to(beta, y.shape))


def test_layernorm_matches_torch_float64():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((500, 128)) + 0.5).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    beta = (rng.standard_normal(128) * 0.1).astype(np.float32)
    y = oracle.layernorm(x, gamma, beta, 1e-6)
    ref = torch.nn.functional.layer_norm(
        torch.from_numpy(x).double(), (128,), torch.from_numpy(gamma).double(),
        torch.from_numpy(beta).double(), eps=1e-6).float().numpy()
    ulp = np.spacing(np.abs(ref))
    assert np.all(np.abs(y - ref) <= ulp)


def test_hadamard_matches_scipy_and_is_an_involution():
    from scipy.linalg import hadamard as sylvester
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((64, 128)) * 5).astype(np.float32)
    y = oracle.hadamard(x)
    ref = x.astype(np.float64) @ sylvester(128).T / np.sqrt(128.0)
    scale = np.abs(x).sum(axis=1, keepdims=True) / np.sqrt(128.0)
    assert np.all(np.abs(y - ref) <= 8 * 2.0 ** -24 * scale)
    # orthonormal and symmetric: applying it twice gives x back, norms are kept
    assert np.allclose(oracle.hadamard(y), x, rtol=0, atol=1e-5 * np.abs(x).max())
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-6)


def test_hadamard_of_unit_vectors():
    """H e_j / sqrt(128) is the j-th Sylvester column scaled: entries +-2^-3.5."""
    x = np.eye(128, dtype=np.float32)[[0, 1, 77]]
    y = oracle.hadamard(x)
    s = np.float32(1.0 / np.sqrt(128.0))
    assert np.all(np.abs(y) == s)
    assert np.all(y[0] == s)
    assert np.array_equal(y[1], np.where(np.arange(128) & 1, -s, s).astype(np.float32))
