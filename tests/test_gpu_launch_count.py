"""One kernel launch per call: each entry point is captured alone into a CUDA
graph on a raw stream (runtime API through ctypes) and the graph's nodes are
counted -- the fused call, on either kernel, and the k-only and logits calls
give one node; the unfused chain gives its four."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _gpu import new_cache, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
            break
        except OSError:
            lib = None
    if lib is None:
        pytest.skip("the CUDA runtime library is not loadable by name")
    return lib


def _nodes(rt, launch):
    """Capture launch(stream_handle) alone and count the graph's nodes."""
    torch.cuda.synchronize()
    stream = ctypes.c_void_p()
    assert rt.cudaStreamCreateWithFlags(ctypes.byref(stream), 1) == 0  # non-blocking
    graph = ctypes.c_void_p()
    try:
        assert rt.cudaStreamBeginCapture(stream, 1) == 0  # thread-local capture mode
        launch(stream.value)
        assert rt.cudaStreamEndCapture(stream, ctypes.byref(graph)) == 0
        n = ctypes.c_size_t(0)
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        return n.value
    finally:
        if graph.value:
            rt.cudaGraphDestroy(graph)
        rt.cudaStreamDestroy(stream)


def _qk_call(inp, d, cache, q_out, w_out, **kw):
    import prep_token_gb300 as dp
    return lambda s: dp.dsa_indexer_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        q_fp8_out=q_out, weights_out=w_out, max_position=inp.max_position, stream=s, **kw)


@pytest.mark.parametrize("kernel", ["direct", "pipeline"])
@pytest.mark.parametrize("hadamard", [False, True])
def test_fused_call_is_one_launch(rt, kernel, hadamard):
    inp = synth.make_decode(seed=120, T=16, H=8)
    d = to_device(inp)
    cache = new_cache(inp)
    q_out = torch.empty((16, 8, 128), dtype=torch.uint8, device="cuda")
    w_out = torch.empty((16, 8), dtype=torch.float32, device="cuda")
    call = _qk_call(inp, d, cache, q_out, w_out, kernel=kernel, hadamard=hadamard)
    call(torch.cuda.current_stream().cuda_stream)  # first call sets up the device, outside capture
    assert _nodes(rt, call) == 1


def test_k_only_and_unfused_launch_counts(rt):
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=121, T=16, H=8)
    d = to_device(inp)
    cache = new_cache(inp)

    def k_only(s):
        dp.dsa_indexer_k_prepare_store(
            d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
            inp.eps, cache, inp.page_size, inp.rope_dim, inp.style,
            max_position=inp.max_position, stream=s)

    ws = torch.empty(dp.dsa_unfused_workspace_bytes(16, 8), dtype=torch.uint8, device="cuda")
    q_out = torch.empty((16, 8, 128), dtype=torch.uint8, device="cuda")
    w_out = torch.empty((16, 8), dtype=torch.float32, device="cuda")

    def unfused(s):
        dp.dsa_indexer_qk_prepare_store_unfused(
            d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim,
            inp.style, q_fp8_out=q_out, weights_out=w_out, workspace=ws,
            max_position=inp.max_position, stream=s)

    for f in (k_only, unfused):
        f(torch.cuda.current_stream().cuda_stream)
    assert _nodes(rt, k_only) == 1
    assert _nodes(rt, unfused) == 4


def test_logits_call_is_one_launch(rt):
    import prep_token_gb300 as dp
    li = synth.make_logits(seed=122, T=4, H=16, context=300)
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, w, cache, bt, lens = dv(li.q_fp8), dv(li.weights), dv(li.cache), dv(li.block_table), dv(li.context_lens)
    out = torch.empty((li.T, li.max_context), dtype=torch.float32, device="cuda")

    def call(s):
        dp.dsa_indexer_mqa_logits(q, w, cache, li.page_size, bt, lens, li.max_context,
                                  logits=out, stream=s)

    call(torch.cuda.current_stream().cuda_stream)
    assert _nodes(rt, call) == 1
