"""The no-allocation entry point of the unfused chain, through the C ABI.

Some callers cannot allocate device memory when they run the chain -- an
engine whose pool owns the whole GPU, a plugin that is only handed input and
output pointers -- so this entry point keeps the chain's bf16 intermediates in
a buffer compiled into the library instead of a caller workspace.  Its output
must match the workspace entry point's on two calls in a row (the second call
finds the first call's data still in the buffer).  This file sorts last so a
run that stops at the first failure has run everything else before it.
"""
import numpy as np
import pytest
import torch

import synth
from _compare import compare
from _gpu import SENTINEL, new_cache, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _outputs(inp):
    return (torch.empty((inp.T, inp.H, 128), dtype=torch.float8_e4m3fn, device="cuda"),
            torch.empty((inp.T, inp.H), dtype=torch.float32, device="cuda"), new_cache(inp))


def _call(fn, inp, d, q_out, w_out, cache, **kw):
    fn(d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
       d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
       q_fp8_out=q_out, weights_out=w_out, max_position=inp.max_position, **kw)
    torch.cuda.synchronize()
    return dict(q_fp8=q_out.view(torch.uint8).cpu().numpy(), weights=w_out.cpu().numpy(),
                cache=cache.cpu().numpy())


@pytest.mark.parametrize("shape", [(64, 64, synth.GPTJ), (256, 32, synth.NEOX)])
def test_noalloc_matches_workspace_entry_on_two_calls(shape):
    import prep_token_gb300 as dp
    T, H, style = shape
    for seed in (41, 42):   # two calls in a row on different data
        inp = synth.make_decode(seed=seed, T=T, H=H, style=style)
        d = to_device(inp)
        ref = _call(dp.dsa_indexer_qk_prepare_store_unfused, inp, d, *_outputs(inp))
        got = _call(dp.dsa_indexer_qk_prepare_store_unfused_noalloc, inp, d, *_outputs(inp))
        rep = compare(inp, got, ref)
        assert rep["ok"], rep
        for key in ("q_fp8", "weights", "cache"):
            assert np.array_equal(got[key], ref[key]), key


def test_noalloc_rejects_calls_beyond_its_buffer():
    import prep_token_gb300 as dp
    inp = synth.make_prefill(T=2048, H=64)   # 2048 * 66 * 256 B > 32 MiB
    d = to_device(inp)
    q_out, w_out, cache = _outputs(inp)
    with pytest.raises(dp.DsaError) as exc:
        _call(dp.dsa_indexer_qk_prepare_store_unfused_noalloc, inp, d, q_out, w_out, cache)
    assert exc.value.status == 6
    assert torch.all(cache == SENTINEL)


def test_noalloc_at_its_exact_limit():
    """T * (H + 2) * 256 bytes equal to the 32 MiB buffer: accepted, and the
    same bytes as the workspace entry point."""
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=43, T=2048, H=62, style=synth.NEOX)
    assert dp.dsa_unfused_workspace_bytes(inp.T, inp.H) == 32 << 20
    d = to_device(inp)
    ref = _call(dp.dsa_indexer_qk_prepare_store_unfused, inp, d, *_outputs(inp))
    got = _call(dp.dsa_indexer_qk_prepare_store_unfused_noalloc, inp, d, *_outputs(inp))
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(got[key], ref[key]), key


def test_noalloc_two_pdl_calls_in_a_row():
    """Two calls with programmatic dependent launch back to back on one
    stream share the buffer in turn (each launch waits for the one before):
    both give the eager bytes."""
    import prep_token_gb300 as dp
    a = synth.make_decode(seed=44, T=64, H=64)
    b = synth.make_decode(seed=45, T=64, H=64)
    da, db = to_device(a), to_device(b)
    ref_a = _call(dp.dsa_indexer_qk_prepare_store_unfused, a, da, *_outputs(a))
    ref_b = _call(dp.dsa_indexer_qk_prepare_store_unfused, b, db, *_outputs(b))
    outs_a, outs_b = _outputs(a), _outputs(b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for inp, d, (q_out, w_out, cache) in ((a, da, outs_a), (b, db, outs_b)):
            dp.dsa_indexer_qk_prepare_store_unfused_noalloc(
                d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"],
                d["gamma"], d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size,
                inp.rope_dim, inp.style, q_fp8_out=q_out, weights_out=w_out,
                max_position=inp.max_position, pdl=True, stream=s)
    s.synchronize()
    for ref, (q_out, w_out, cache) in ((ref_a, outs_a), (ref_b, outs_b)):
        assert np.array_equal(q_out.view(torch.uint8).cpu().numpy(), ref["q_fp8"])
        assert np.array_equal(w_out.cpu().numpy(), ref["weights"])
        assert np.array_equal(cache.cpu().numpy(), ref["cache"])
