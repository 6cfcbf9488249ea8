"""GPU scales at the exact ue8m0 boundaries, against the oracle.

The scale exponent is the smallest integer e with max(amax, 1e-4) <= 448 * 2^e
(vllm PR "[ROCm][Perf] Enable fused indexer-Q RoPE+quant kernel for
DeepSeek/GLM sparse attention", Kernel-level evidence, "q -> FP8 (ue8m0)
quant"; sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant +
K-cache write", Accuracy: ue8m0 scales identical).  amax = 448 * 2^k gives
e = k and the next representable value above it gives k + 1; amax at or below
the 1e-4 floor gives e = -22 whatever it is (448 * 2^-23 < 1e-4 <= 448 * 2^-22).

Keys reach the quantiser in fp32: a constant key row has LayerNorm output
exactly beta (x - mean is 0, so the affine step returns beta), and position 0
makes RoPE the identity (cos 1, sin 0).  A planted beta therefore puts any
fp32 value -- a boundary and its fp32 neighbours, 1e-4 and its neighbours --
into the quantiser as the key's amax.  Queries are bf16 and also at position
0, so their amax is a planted bf16 value: a boundary and its bf16
neighbours, values below the floor, all-zero rows.

Every case runs through the direct kernel, the pipeline kernel and the
k-only kernels, in both pairings, plain and with the Hadamard rotation (whose
rotated amax is not planted, but must still match the oracle bit for bit),
and checks the oracle's exponents against the definition above."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from _compare import assert_parity
from _gpu import run_k, run_qk, to_device
from _run import run_oracle_qk

pytestmark = pytest.mark.gpu

D = 128
T, H, ROPE = 16, 8, 64
FLOOR = float(np.float32(1e-4))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


def expected_exp(amax: float) -> int:
    """The smallest e with max(amax, 1e-4f) <= 448 * 2^e, in exact arithmetic."""
    a = max(Fraction(amax), Fraction(FLOOR))
    e = -160
    while a > 448 * Fraction(2) ** e:
        e += 1
    return e


def f32_next(x, direction):
    return float(np.nextafter(np.float32(x), np.float32(direction)))


def bf16_neighbours(x):
    """x (bf16-exact) and the bf16 values just below and above it."""
    b = int(synth.to_bf16_bits(np.array([x], np.float32))[0])
    vals = [synth.bf16_bits_to_f32(np.array([b + d], np.uint16))[0] for d in (-1, 0, 1)]
    return [float(v) for v in vals]


def key_targets():
    out = []
    for k in (-22, -10, 0, 7):
        b = 448.0 * 2.0 ** k
        out += [b, f32_next(b, np.inf), f32_next(b, 0.0)]
    out += [FLOOR, f32_next(FLOOR, np.inf), f32_next(FLOOR, 0.0), 448.0 * 2.0 ** -23, 0.0]
    return out


def query_targets():
    out = [0.0, 448.0 * 2.0 ** -23]
    for k in (-22, -5, 0, 3, 8):
        out += bf16_neighbours(448.0 * 2.0 ** k)
    out += bf16_neighbours(float(synth.bf16_bits_to_f32(synth.to_bf16_bits(
        np.array([FLOOR], np.float32)))[0]))
    return out


def make_case(style, k_target, seed):
    """T tokens at position 0 with constant key rows and beta planted at
    k_target; the query head rows cycle through query_targets(), each with one
    pass-through element at +-target and the rest at most target / 4."""
    rng = np.random.default_rng(seed)
    targets = query_targets()
    q = np.zeros((T * H, D), np.float32)
    for i in range(T * H):
        t = targets[i % len(targets)]
        if t == 0.0:
            continue
        row = (rng.uniform(-0.25, 0.25, D) * t).astype(np.float32)
        row[rng.integers(ROPE, D)] = t * rng.choice([-1.0, 1.0])
        q[i] = row
    qb = synth.to_bf16_bits(q)
    # the planted values are bf16-exact, so rounding keeps every row's amax
    assert np.array_equal(np.abs(synth.bf16_bits_to_f32(qb)).max(axis=1),
                          np.array([targets[i % len(targets)] for i in range(T * H)], np.float32))
    beta = (rng.uniform(-0.25, 0.25, D) * k_target).astype(np.float32)
    if k_target != 0.0:
        beta[rng.integers(0, D)] = np.float32(k_target) * np.float32(rng.choice([-1.0, 1.0]))
    assert np.abs(beta).max() == np.float32(k_target)
    gamma = rng.uniform(0.5, 1.5, D).astype(np.float32)
    k = np.repeat(rng.standard_normal((T, 1)).astype(np.float32), D, axis=1)
    w = rng.standard_normal((T, H)).astype(np.float32)
    kw = np.zeros((T, D + H), np.uint16)
    kw[:, :D] = synth.to_bf16_bits(k)
    kw[:, D:] = synth.to_bf16_bits(w)
    cos, sin = synth.rope_table(16, ROPE)
    slots = rng.choice(4 * 64, size=T, replace=False).astype(np.int64)
    return synth.Inputs(name="ue8m0_boundary", T=T, H=H, rope_dim=ROPE, style=style,
                        page_size=64, num_pages=4, max_position=16,
                        q=qb.reshape(T, H, D), k=kw[:, :D], w=kw[:, D:],
                        positions=np.zeros(T, np.int64), slots=slots, cos=cos, sin=sin,
                        gamma=gamma, beta=beta, kw=kw)


def test_expected_exponent_definition():
    """The helper itself, on values the definition fixes by hand."""
    assert expected_exp(448.0) == 0
    assert expected_exp(f32_next(448.0, np.inf)) == 1
    assert expected_exp(f32_next(448.0, 0.0)) == 0
    assert expected_exp(0.0) == -22
    assert expected_exp(448.0 * 2.0 ** -23) == -22
    assert expected_exp(448.0 * 2.0 ** -22) == -22
    assert expected_exp(f32_next(448.0 * 2.0 ** -22, np.inf)) == -21


@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
@pytest.mark.parametrize("k_target", key_targets())
def test_boundaries(style, k_target):
    inp = make_case(style, k_target, seed=int(abs(k_target) * 1e6) % 10007 + style)
    d = to_device(inp)
    for hadamard in (False, True):
        ref = run_oracle_qk(inp, hadamard=hadamard)
        if not hadamard:
            want_q = np.array([[expected_exp(float(np.abs(synth.bf16_bits_to_f32(inp.q[t, h])).max()))
                                for h in range(H)] for t in range(T)])
            assert np.array_equal(ref["q_exp"], want_q), "oracle q exponents"
            assert np.all(ref["k_exp"] == expected_exp(k_target)), "oracle k exponents"
        first = None
        for kern in ("direct", "pipeline"):
            gpu = run_qk(inp, d, kernel=kern, hadamard=hadamard)
            assert_parity(inp, gpu, ref)
            assert np.array_equal(gpu["cache"], ref["cache"]), f"cache bytes ({kern}, {hadamard})"
            gk = run_k(inp, d, kernel=kern, hadamard=hadamard)
            assert np.array_equal(gk["cache"], ref["cache"]), f"k-only cache ({kern}, {hadamard})"
            if first is None:
                first = gpu
            else:
                assert np.array_equal(gpu["q_fp8"], first["q_fp8"])
