"""Pins of the oracle's fp8 paged MQA logits (the consumer of the index-K
cache): a hand-worked case, a float64 brute force with CPU torch's e4m3
decode, the ReLU identity relu(x) - relu(-x) = x, linearity in the weights,
the context mask, and invariance under a consistent relabelling of pages."""
import numpy as np
import torch

import oracle
import synth


def _decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def _brute(li):
    cache = li.cache.reshape(li.num_pages, -1)
    P = li.page_size
    out = np.full((li.T, li.max_context), -np.inf)
    q = _decode(li.q_fp8)
    for t in range(li.T):
        for j in range(li.context_lens[t]):
            page = cache[li.block_table[t, j // P]]
            k = _decode(page[(j % P) * 128:(j % P + 1) * 128])
            scale = page[P * 128:].view(np.float32)[j % P]
            dots = q[t] @ k
            out[t, j] = scale * np.sum(li.weights[t].astype(np.float64) * np.maximum(dots, 0))
    return out


def test_hand_worked_case():
    # H = 1; q = 1.0 (0x38) at d = 0; key 0 = 2.0 (0x40) at d = 0 with scale 0.5;
    # key 1 = -2.0 (0xC0): weight 3 gives 0.5 * 3 * max(1 * 2, 0) = 3 and 0.
    P = 4
    cache = np.zeros((1, P * 132), np.uint8)
    cache[0, 0] = 0x40
    cache[0, 128] = 0xC0
    cache[0, P * 128:].view(np.float32)[:] = 0.5
    q = np.zeros((1, 1, 128), np.uint8)
    q[0, 0, 0] = 0x38
    err, out = oracle.mqa_logits(q, np.array([[3.0]], np.float32), cache.reshape(-1), 1, P,
                                 np.zeros((1, 1), np.int32), np.array([2], np.int32), 4)
    assert err == 0
    assert list(out[0]) == [3.0, 0.0, -np.inf, -np.inf]


def test_bruteforce_small():
    li = synth.make_logits(seed=1, T=3, H=4, context=150, page_size=64, ragged=True)
    err, out = oracle.mqa_logits(li.q_fp8, li.weights, li.cache, li.num_pages, li.page_size,
                                 li.block_table, li.context_lens, li.max_context)
    ref = _brute(li)
    assert err == 0
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(out), fin)
    assert np.all(np.abs(out[fin] - ref[fin]) <= 1e-6 * np.abs(ref[fin]) + 1e-30)


def test_relu_identity_and_linearity():
    li = synth.make_logits(seed=2, T=2, H=8, context=128, page_size=64)
    args = (li.cache, li.num_pages, li.page_size, li.block_table, li.context_lens,
            li.max_context)
    _, pos = oracle.mqa_logits(li.q_fp8, li.weights, *args)
    _, neg = oracle.mqa_logits(li.q_fp8 ^ np.uint8(0x80), li.weights, *args)
    _, dbl = oracle.mqa_logits(li.q_fp8, li.weights * 2, *args)
    assert np.array_equal(dbl, pos * 2)
    # relu(x) - relu(-x) = x: the difference is linear in q, so it must equal
    # the plain weighted dot product
    cache = li.cache.reshape(li.num_pages, -1)
    q = _decode(li.q_fp8)
    for t in range(li.T):
        for j in range(0, 128, 17):
            page = cache[li.block_table[t, j // 64]]
            k = _decode(page[(j % 64) * 128:(j % 64 + 1) * 128])
            scale = page[64 * 128:].view(np.float32)[j % 64]
            lin = scale * np.sum(li.weights[t] * (q[t] @ k))
            assert abs((pos[t, j] - neg[t, j]) - lin) <= 1e-5 * (abs(pos[t, j]) + abs(neg[t, j]) + 1e-30)


def test_page_relabelling_is_invisible():
    li = synth.make_logits(seed=3, T=2, H=4, context=200, page_size=64, ragged=True, spare_pages=3)
    _, a = oracle.mqa_logits(li.q_fp8, li.weights, li.cache, li.num_pages, li.page_size,
                             li.block_table, li.context_lens, li.max_context)
    rng = np.random.default_rng(0)
    perm = rng.permutation(li.num_pages)           # new label of old page p is perm[p]
    cache = li.cache.reshape(li.num_pages, -1)
    moved = np.empty_like(cache)
    moved[perm] = cache
    table = perm[li.block_table].astype(np.int32)
    _, b = oracle.mqa_logits(li.q_fp8, li.weights, moved.reshape(-1), li.num_pages, li.page_size,
                             table, li.context_lens, li.max_context)
    assert np.array_equal(a, b)
    assert np.all(np.isneginf(a[np.arange(a.shape[1])[None, :] >= li.context_lens[:, None]]))
