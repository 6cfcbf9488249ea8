"""The unfused four-launch chain (LayerNorm, RoPE, q quant + fold, k quant +
store, bf16 between launches) through the C ABI, against the oracle's chain
mode: q codes exact, scales and slots exact, k codes within one step in at
most 0.1% of elements, weights within 1e-6."""
import numpy as np
import pytest
import torch

import synth
from _compare import assert_parity
from _gpu import SENTINEL, new_cache, to_device
from _run import run_oracle_qk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


def run_unfused(inp, d, cache=None, err=None, **kw):
    import prep_token_gb300 as dp
    kw.setdefault("cache_layout", "token_major" if inp.token_major else "paged")
    cache = new_cache(inp) if cache is None else cache
    q_fp8, weights = dp.dsa_indexer_qk_prepare_store_unfused(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        err_flags=err, max_position=inp.max_position, **kw)
    torch.cuda.synchronize()
    return dict(q_fp8=q_fp8.view(torch.uint8).cpu().numpy(), weights=weights.cpu().numpy(),
                cache=cache.cpu().numpy())


def _check(inp):
    d = to_device(inp)
    return assert_parity(inp, run_unfused(inp, d), run_oracle_qk(inp, chain=True))


@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_tiny(style):
    _check(synth.make_tiny(style=style))


def test_decode():
    _check(synth.make_decode())


@pytest.mark.parametrize("T", [1, 64, 256])
def test_sweep(T):
    _check(synth.make_sweep(T))


def test_prefill_full_size():
    _check(synth.make_prefill())


@pytest.mark.parametrize("T,H", [(3, 5), (33, 13), (517, 100), (5, 128)])
def test_ragged(T, H):
    _check(synth.make_decode(seed=T * 7 + H, T=T, H=H, style=(T + H) % 2))


@pytest.mark.parametrize("rope_dim", [0, 16, 32, 128])
@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_rope_dims(rope_dim, style):
    inp = synth.make_decode(seed=rope_dim + 3, T=24, H=6, style=style)
    inp.cos, inp.sin = synth.rope_table(inp.max_position, max(rope_dim, 16))
    inp.rope_dim = rope_dim
    _check(inp)


def test_error_bits_and_workspace_reuse():
    inp = synth.make_decode(seed=31, T=20, H=4)
    inp.positions = inp.positions.copy()
    inp.slots = inp.slots.copy()
    inp.positions[2] = inp.max_position
    inp.slots[4] = -1
    d = to_device(inp)
    import prep_token_gb300 as dp
    ws = torch.full((dp.dsa_unfused_workspace_bytes(inp.T, inp.H),), 0x7F, dtype=torch.uint8,
                    device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_unfused(inp, d, err=err, workspace=ws)
    assert int(err.item()) == 3
    ref = run_oracle_qk(inp, chain=True)
    assert ref["err"] == 3
    ok = np.ones(inp.T, bool)
    ok[2] = False
    from _compare import compare
    rep = compare(inp, dict(q_fp8=got["q_fp8"][ok], weights=got["weights"][ok], cache=got["cache"]),
                  dict(q_fp8=ref["q_fp8"][ok], weights=ref["weights"][ok], cache=ref["cache"]))
    assert rep["ok"], rep
    # a second call on the same (now dirty) workspace gives the same bytes
    again = run_unfused(inp, d, workspace=ws)
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(np.asarray(again[key])[ok] if key != "cache" else again[key],
                              np.asarray(got[key])[ok] if key != "cache" else got[key]), key


def test_pdl_graph_matches_eager():
    inp = synth.make_decode(seed=32, T=64, H=64)
    d = to_device(inp)
    eager = run_unfused(inp, d)
    import prep_token_gb300 as dp
    cache = new_cache(inp)
    ws = torch.empty(dp.dsa_unfused_workspace_bytes(64, 64), dtype=torch.uint8, device="cuda")
    q_out = torch.empty((64, 64, 128), dtype=torch.float8_e4m3fn, device="cuda")
    w_out = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            dp.dsa_indexer_qk_prepare_store_unfused(
                d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"],
                d["gamma"], d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size,
                inp.rope_dim, inp.style, q_fp8_out=q_out, weights_out=w_out, workspace=ws,
                max_position=inp.max_position, pdl=True, stream=s)
    cache.fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(q_out.view(torch.uint8).cpu().numpy(), eager["q_fp8"])
    assert np.array_equal(w_out.cpu().numpy(), eager["weights"])
    assert np.array_equal(cache.cpu().numpy(), eager["cache"])


@pytest.mark.parametrize("page_size", [1, 64])
def test_token_major_cache_layout(page_size):
    inp = synth.make_decode(seed=60 + page_size, T=50, H=8)
    inp.page_size, inp.num_pages = page_size, (4096 * 64) // page_size
    inp.token_major = True
    _check(inp)
