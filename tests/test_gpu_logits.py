"""fp8 paged MQA logits on the tensor cores, through the C ABI, against the
oracle.  Tolerance, from the arithmetic: every e4m3 x e4m3 product is exact
in fp32; the kernel adds the 128 products of a dot product in fp32 on the
tensor cores, then the H weighted ReLU terms in fp32, and scales once, so
|gpu - ref| <= (128 + H + 4) * 2^-24 * k_scale * sum_h |w_h| * sum_d |q_hd k_d|
(the first-order rounding bound of those sums); masked columns must be
exactly -inf."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


def _decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def _tolerance(li, tokens):
    """(128 + H + 4) 2^-24 k_scale sum_h |w_h| sum_d |q_hd k_d| per (token, key)."""
    cache = li.cache.reshape(li.num_pages, -1)
    P = li.page_size
    tol = np.zeros((len(tokens), li.max_context))
    for r, t in enumerate(tokens):
        n = min(int(li.context_lens[t]), li.max_context)
        pages = cache[li.block_table[t, :(n + P - 1) // P]]
        kc = pages[:, :P * 128].reshape(-1, 128)[:n]
        ks = np.ascontiguousarray(pages[:, P * 128:]).view(np.float32).reshape(-1)[:n]
        mass = np.abs(_decode(li.q_fp8[t])) @ np.abs(_decode(kc)).T       # [H, n]
        tol[r, :n] = (128 + li.H + 4) * 2.0 ** -24 * ks * (
            np.abs(li.weights[t].astype(np.float64)) @ mass)
    return tol


def _run_gpu(li, err=None):
    import prep_token_gb300 as dp
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = dp.dsa_indexer_mqa_logits(d(li.q_fp8), d(li.weights), d(li.cache), li.page_size,
                                    d(li.block_table), d(li.context_lens), li.max_context,
                                    err_flags=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle(li, tokens, expect_err=0):
    sub = synth.LogitsInputs(
        T=len(tokens), H=li.H, page_size=li.page_size, num_pages=li.num_pages,
        q_fp8=np.ascontiguousarray(li.q_fp8[tokens]), weights=np.ascontiguousarray(li.weights[tokens]),
        cache=li.cache, block_table=np.ascontiguousarray(li.block_table[tokens]),
        context_lens=np.ascontiguousarray(li.context_lens[tokens]), max_context=li.max_context)
    err, out = oracle.mqa_logits(sub.q_fp8, sub.weights, sub.cache, sub.num_pages, sub.page_size,
                                 sub.block_table, sub.context_lens, sub.max_context)
    assert err == expect_err
    return out


def _check(li, tokens=None, err=None):
    tokens = list(range(li.T)) if tokens is None else tokens
    got = _run_gpu(li, err=err)[tokens]
    ref = _oracle(li, tokens)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "masked columns differ"
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN columns (bad pages) differ"
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    tol = _tolerance(li, tokens)[fin] + 1e-30
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert np.all(err <= tol), f"max err/tol {worst}"
    return worst


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_small_ragged(H):
    li = synth.make_logits(seed=H, T=3, H=H, context=300, ragged=True, spare_pages=2)
    _check(li)


def test_partial_tiles_and_empty_context():
    li = synth.make_logits(seed=7, T=4, H=64, context=129)
    li.context_lens = np.array([0, 1, 64, 129], np.int32)
    li.max_context = 200
    # the binding wants a table that covers max_context (padding entries unused)
    li.block_table = np.pad(li.block_table, ((0, 0), (0, 4 - li.block_table.shape[1])))
    _check(li)


def test_decode_full_size_all_tokens():
    """64 sequences x 16384 keys x 64 heads (the decode step at 16K context):
    every column of every token against the oracle."""
    li = synth.make_logits(seed=9, T=64, H=64, context=16384)
    worst = _check(li)
    print("max err/tol", worst)


def test_decode_full_size_ragged():
    """The same step with context lengths uniform in [1, 16384]: each token's
    tiles end at its own length (the last one part-filled), every column
    beyond it is -inf, and the CTAs of short tokens have no tiles at all."""
    li = synth.make_logits(seed=11, T=64, H=64, context=16384, ragged=True)
    assert li.context_lens.min() < 4096 and li.max_context > 12288
    worst = _check(li)
    print("max err/tol", worst)


def test_bad_page_sets_error_bit_and_nan_columns():
    """A block-table entry outside [0, num_pages) sets the error bit, and the
    64 columns of that block are NaN, as in the oracle; every other column
    of both tokens still matches."""
    li = synth.make_logits(seed=10, T=2, H=16, context=200)
    li.block_table = li.block_table.copy()
    li.block_table[1, 0] = li.num_pages + 5
    li.block_table[0, 2] = -3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run_gpu(li, err=err)
    assert int(err.item()) & 2
    ref = _oracle(li, [0, 1], expect_err=2)
    assert np.isnan(ref[1, :64]).all() and np.isnan(ref[0, 128:192]).all()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = np.isfinite(ref)
    assert np.all(np.abs(got[fin] - ref[fin]) <= _tolerance_safe(li, [0, 1])[fin] + 1e-30)


def _tolerance_safe(li, tokens):
    """_tolerance with out-of-range block-table entries read as page 0 (their
    columns are compared for NaN only)."""
    saved = li.block_table
    li.block_table = np.where((saved < 0) | (saved >= li.num_pages), 0, saved).astype(saved.dtype)
    try:
        return _tolerance(li, tokens)
    finally:
        li.block_table = saved


@pytest.mark.parametrize("pdl", [True, "early"])
def test_pdl_graph_matches_eager(pdl):
    """A graph of PDL launches (with early reads of the block table and the
    context lengths, which no kernel in the graph writes) gives the eager
    bytes."""
    import prep_token_gb300 as dp
    li = synth.make_logits(seed=11, T=8, H=64, context=1000, ragged=True)
    eager = _run_gpu(li)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, w, cache, bt, lens = d(li.q_fp8), d(li.weights), d(li.cache), d(li.block_table), d(li.context_lens)
    out = torch.full((li.T, li.max_context), 7.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dp.dsa_indexer_mqa_logits(q, w, cache, li.page_size, bt, lens, li.max_context,
                                  logits=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            dp.dsa_indexer_mqa_logits(q, w, cache, li.page_size, bt, lens, li.max_context,
                                      logits=out, pdl=pdl, stream=s)
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(eager))
    fin = np.isfinite(eager)
    assert np.array_equal(got[fin], eager[fin])


def test_context_longer_than_max_context_is_clamped():
    """Columns exist only below max_context: a longer context is clamped to it
    (no wait is left hanging, no error bit), as the oracle defines."""
    li = synth.make_logits(seed=12, T=3, H=32, context=600)
    li.context_lens = np.array([600, 130, 0], np.int32)
    li.max_context = 256
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run_gpu(li, err=err)
    assert int(err.item()) == 0
    ref = _oracle(li, [0, 1, 2])
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), ~fin)
    assert np.all(np.abs(got[fin] - ref[fin]) <= _tolerance(li, [0, 1, 2])[fin] + 1e-30)


def test_binding_rejects_tensors_on_the_wrong_device_or_short_tables():
    import prep_token_gb300 as dp
    li = synth.make_logits(seed=13, T=2, H=16, context=200)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = [d(li.q_fp8), d(li.weights), d(li.cache), li.page_size, d(li.block_table),
            d(li.context_lens), li.max_context]
    bad = list(args)
    bad[1] = torch.from_numpy(np.ascontiguousarray(li.weights))  # weights on the host
    with pytest.raises(ValueError):
        dp.dsa_indexer_mqa_logits(*bad)
    bad = list(args)
    bad[4] = args[4][:, :1]  # one 64-key block cannot cover max_context = 200
    with pytest.raises(ValueError):
        dp.dsa_indexer_mqa_logits(*bad)
    with pytest.raises(ValueError):
        dp.dsa_indexer_mqa_logits(*args, err_flags=torch.zeros(1, dtype=torch.int32))
