"""The shared input generator: determinism, layout and the planted structure
of the stress workload (checked with the oracle where it needs the path)."""
import numpy as np

import synth
from _run import run_oracle_qk


def test_deterministic_and_distinct_slots():
    a, b = synth.make_decode(T=64, H=8), synth.make_decode(T=64, H=8)
    for key in ("q", "k", "w", "positions", "slots", "cos", "sin", "gamma", "beta"):
        assert np.array_equal(getattr(a, key), getattr(b, key)), key
    assert np.unique(a.slots).size == a.T
    assert a.slots.max() < a.num_pages * a.page_size
    assert a.positions.max() < a.max_position


def test_fused_kw_layout():
    inp = synth.make_decode(T=16, H=64)
    assert inp.kw.shape == (16, 192)
    assert inp.k_stride_t == 192 and inp.w_stride_t == 192
    assert np.array_equal(inp.kw[:, :128], inp.k) and np.array_equal(inp.kw[:, 128:], inp.w)
    k = synth.bf16_bits_to_f32(inp.k)
    assert 0.3 < k.mean() < 0.7  # k ~ N(0,1) + 0.5


def test_prefill_layout():
    inp = synth.make_prefill(T=256, H=4)
    assert np.array_equal(inp.positions, np.arange(256))
    assert np.array_equal(inp.slots, np.arange(256)) and inp.num_pages == 4


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.0 - 2 ** -7], np.float32)
    got = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    assert list(got) == [1.0, 1.0 + 2 ** -6, 1.0, -2.0]


def test_stress_planted_structure():
    inp = synth.make_stress(n_seq=2, seq_len=128, H=8, pages=16)
    T = inp.T
    assert T == 256
    # slots: a permutation of whole pages, 64 consecutive tokens per page
    assert np.unique(inp.slots).size == T
    assert np.all(inp.slots.reshape(-1, 64) // 64 == (inp.slots.reshape(-1, 64) // 64)[:, :1])
    assert np.array_equal(inp.positions, np.tile(np.arange(128), 2))
    q = inp.q.reshape(T * 8, 128)
    assert np.all(q[inp.zero_q_rows] == 0) and inp.zero_q_rows.size >= 1
    assert np.all(inp.k[inp.zero_k_rows] == 0) and inp.zero_k_rows.size >= 1
    # planted rows: the oracle's scale is the planted one, and about 1% of all q
    # elements are exact E4M3 midpoints at that scale
    out = run_oracle_qk(inp)
    assert out["err"] == 0
    qe = out["q_exp"].reshape(-1)
    assert np.array_equal(qe[inp.planted_rows], inp.planted_exp)
    mids = set(synth.e4m3_midpoints().tolist())
    qf = synth.bf16_bits_to_f32(q[inp.planted_rows, 64:]).astype(np.float64)
    scaled = np.abs(qf) * np.exp2(-inp.planted_exp)[:, None]
    n_mid = sum(v in mids for v in scaled.reshape(-1).tolist())
    frac = n_mid / q.size
    # ~1% planted, plus the ties bf16 data hits by itself (a bf16 value scaled
    # by a power of two is an E4M3 midpoint 1 time in 16)
    assert 0.008 < frac < 0.03, frac
