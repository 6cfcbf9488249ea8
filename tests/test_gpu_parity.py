"""CUDA path vs the oracle, through the C ABI, on every workload shape:
tiny, decode (GPT-J), the decode sweep, prefill and the heavy-tailed stress
set at full size, plus ragged shapes, strided views, rope-cache replacement,
the live-token slice, device error bits and CUDA-graph replay."""
import numpy as np
import pytest
import torch

import synth
from _compare import assert_parity, compare
from _gpu import SENTINEL, new_cache, run_k, run_qk, to_device
from _run import cache_views, run_oracle_k, run_oracle_qk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


KERNELS = ("direct", "pipeline")


def _check(inp, q_exact=True, kernels=KERNELS):
    """Every kernel must match the oracle, and all of them (fused and k-only)
    must write the same bytes."""
    d = to_device(inp)
    ref = run_oracle_qk(inp)
    first = None
    for kern in kernels:
        gpu = run_qk(inp, d, kernel=kern)
        rep = assert_parity(inp, gpu, ref, q_exact=q_exact)
        gk = run_k(inp, d, kernel=kern)
        assert np.array_equal(gk["cache"], gpu["cache"]), f"k-only and qk caches differ ({kern})"
        if first is None:
            first = gpu
        else:
            for key in ("q_fp8", "weights", "cache"):
                assert np.array_equal(gpu[key], first[key]), f"{key}: {kern} != {kernels[0]}"
    return rep


@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_tiny(style):
    _check(synth.make_tiny(style=style))


def test_decode_gptj():
    _check(synth.make_decode())


@pytest.mark.parametrize("T", [1, 8, 32, 64, 256])
def test_decode_sweep(T):
    _check(synth.make_sweep(T))


def test_prefill_full_size():
    _check(synth.make_prefill())


@pytest.fixture(scope="module")
def stress_neox():
    return synth.make_stress(style=synth.NEOX)


@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_stress_full_size(stress_neox, style):
    inp = stress_neox
    inp.style = style
    rep = _check(inp)
    print(style, rep)


@pytest.mark.parametrize("H", [1, 3, 5, 7, 13, 64, 100, 128])
@pytest.mark.parametrize("T", [1, 3, 33, 517])
def test_ragged_shapes(T, H):
    _check(synth.make_decode(seed=T * 1000 + H, T=T, H=H, style=(T + H) % 2))


@pytest.mark.parametrize("rope_dim", [0, 16, 32, 64, 128])
@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_rope_dims(rope_dim, style):
    inp = synth.make_decode(seed=rope_dim + 7, T=40, H=6, style=style)
    cos, sin = synth.rope_table(inp.max_position, max(rope_dim, 16))
    inp.rope_dim = rope_dim
    inp.cos, inp.sin = cos, sin
    _check(inp)


@pytest.mark.parametrize("page_size", [4, 12, 16, 64, 100, 256])
def test_page_sizes(page_size):
    inp = synth.make_decode(seed=page_size, T=50, H=4)
    inp.page_size = page_size
    inp.num_pages = (4096 * 64) // page_size
    _check(inp)


def test_strided_equals_contiguous():
    a = synth.make_tiny(seed=9, T=37, H=16, fused_kw=True)
    b = synth.make_tiny(seed=9, T=37, H=16, fused_kw=False)
    da, db = to_device(a), to_device(b)
    ga, gb = run_qk(a, da), run_qk(b, db)
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(ga[key], gb[key]), key
    # q with a padded head stride and padded token stride
    qpad = torch.zeros((37, 16, 192), dtype=torch.bfloat16, device="cuda")
    qpad[:, :, :128] = db["q"]
    dc = dict(db)
    dc["q"] = qpad[:, :, :128]
    assert dc["q"].stride() == (16 * 192, 192, 1)
    gc = run_qk(b, dc)
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(gc[key], gb[key]), key


def test_rope_cache_replaced_between_calls():
    """The library keeps no table pointer or contents: overwrite the cos/sin
    cache in place and the next call follows it."""
    a = synth.make_tiny(seed=10, T=16, H=4)
    d = to_device(a)
    g1 = run_qk(a, d)
    cos2, sin2 = synth.rope_table(a.max_position, 64, base=500000.0)
    d["cos"].copy_(torch.from_numpy(cos2))
    d["sin"].copy_(torch.from_numpy(sin2))
    g2 = run_qk(a, d)
    a.cos, a.sin = cos2, sin2
    assert_parity(a, g2, run_oracle_qk(a))
    assert not np.array_equal(g1["q_fp8"], g2["q_fp8"])


def test_live_token_slice():
    """num_tokens < buffer rows: only the live tokens are read and written."""
    inp = synth.make_decode(seed=11, T=64, H=8)
    d = to_device(inp)
    q_out = torch.full((64, 8, 128), 0x5A, dtype=torch.uint8, device="cuda")
    w_out = torch.full((64, 8), -7.0, dtype=torch.float32, device="cuda")
    cache = new_cache(inp)
    import prep_token_gb300 as dp
    dp.dsa_indexer_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        q_fp8_out=q_out.view(torch.float8_e4m3fn), weights_out=w_out, num_tokens=40,
        max_position=inp.max_position)
    torch.cuda.synchronize()
    ref = run_oracle_qk(inp, T=40)
    got = dict(q_fp8=q_out[:40].cpu().numpy(), weights=w_out[:40].cpu().numpy(),
               cache=cache.cpu().numpy())
    inp40 = synth.make_decode(seed=11, T=64, H=8)
    inp40.T = 40
    assert_parity(inp40, got, ref)
    assert torch.all(q_out[40:] == 0x5A) and torch.all(w_out[40:] == -7.0)


@pytest.mark.parametrize("kernel", ["direct", "pipeline"])
def test_device_error_bits(kernel):
    """Bad positions and slots set their error bits and write nothing, in
    every kernel (k-only with kernel="pipeline" is the k-stream kernel), and
    the other tokens still match the oracle."""
    inp = synth.make_decode(seed=12, T=20, H=4)
    inp.positions = inp.positions.copy()
    inp.slots = inp.slots.copy()
    inp.positions[3] = -1
    inp.positions[5] = inp.max_position
    inp.slots[7] = inp.num_pages * inp.page_size
    inp.slots[9] = -5
    d = to_device(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu = run_qk(inp, d, err=err, kernel=kernel)
    ref = run_oracle_qk(inp)
    assert ref["err"] == 3 and int(err.item()) == 3
    ok = np.ones(inp.T, bool)
    ok[[3, 5]] = False
    # tokens with a bad position write nothing; compare the others
    rep = compare(inp, dict(q_fp8=gpu["q_fp8"][ok], weights=gpu["weights"][ok],
                            cache=gpu["cache"]),
                  dict(q_fp8=ref["q_fp8"][ok], weights=ref["weights"][ok], cache=ref["cache"]))
    assert rep["ok"], rep
    err.zero_()
    gk = run_k(inp, d, err=err, kernel=kernel)
    assert int(err.item()) == 3
    assert np.array_equal(gk["cache"], gpu["cache"])
    err.zero_()
    good = synth.make_decode(seed=12, T=20, H=4)
    run_qk(good, to_device(good), err=err, kernel=kernel)
    run_k(good, to_device(good), err=err, kernel=kernel)
    assert int(err.item()) == 0


def test_cuda_graph_replay_matches_eager():
    inp = synth.make_decode(seed=13, T=64, H=64)
    d = to_device(inp)
    eager = run_qk(inp, d)
    import prep_token_gb300 as dp
    cache = new_cache(inp)
    q_out = torch.empty((64, 64, 128), dtype=torch.float8_e4m3fn, device="cuda")
    w_out = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dp.dsa_indexer_qk_prepare_store(   # warm up outside capture
            d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim,
            inp.style, q_fp8_out=q_out, weights_out=w_out, max_position=inp.max_position)
    torch.cuda.current_stream().wait_stream(s)
    cache.fill_(SENTINEL)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dp.dsa_indexer_qk_prepare_store(
            d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim,
            inp.style, q_fp8_out=q_out, weights_out=w_out, max_position=inp.max_position)
    q_out.view(torch.uint8).zero_()
    cache.fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(q_out.view(torch.uint8).cpu().numpy(), eager["q_fp8"])
    assert np.array_equal(w_out.cpu().numpy(), eager["weights"])
    assert np.array_equal(cache.cpu().numpy(), eager["cache"])
    # new inputs copied into the captured buffers are picked up on replay
    inp2 = synth.make_decode(seed=14, T=64, H=64)
    d2 = to_device(inp2)
    d["q"].copy_(d2["q"])
    d["kw"].copy_(d2["kw"])
    cache.fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    inp2.positions, inp2.slots = inp.positions, inp.slots
    inp2.gamma, inp2.beta = inp.gamma, inp.beta
    got = dict(q_fp8=q_out.view(torch.uint8).cpu().numpy(), weights=w_out.cpu().numpy(),
               cache=cache.cpu().numpy())
    assert_parity(inp2, got, run_oracle_qk(inp2))


def test_empty_call_launches_nothing():
    inp = synth.make_tiny(seed=15)
    d = to_device(inp)
    cache = new_cache(inp)
    import prep_token_gb300 as dp
    q, w = dp.dsa_indexer_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        num_tokens=0, max_position=inp.max_position)
    torch.cuda.synchronize()
    assert q.shape[0] == 0 and w.shape[0] == 0
    assert torch.all(cache == SENTINEL)


def test_pdl_launch_matches():
    """Programmatic dependent launch changes when the kernel may start, not
    what it computes: eager and graph-captured PDL calls give the plain bytes."""
    inp = synth.make_decode(seed=16, T=64, H=64)
    d = to_device(inp)
    plain = run_qk(inp, d)
    for mode in (True, "early"):
        for kern in ("direct", "pipeline"):
            pdl = run_qk(inp, d, pdl=mode, kernel=kern)
            for key in ("q_fp8", "weights", "cache"):
                assert np.array_equal(plain[key], pdl[key]), (key, mode, kern)
    import prep_token_gb300 as dp
    cache = new_cache(inp)
    q_out = torch.empty((64, 64, 128), dtype=torch.float8_e4m3fn, device="cuda")
    w_out = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    k_cache = new_cache(inp)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):   # back-to-back dependent launches inside the graph
            dp.dsa_indexer_qk_prepare_store(
                d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"],
                d["gamma"], d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size,
                inp.rope_dim, inp.style, q_fp8_out=q_out, weights_out=w_out,
                max_position=inp.max_position, pdl="early", stream=s)
            dp.dsa_indexer_k_prepare_store(
                d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
                inp.eps, k_cache, inp.page_size, inp.rope_dim, inp.style,
                max_position=inp.max_position, pdl=True, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(q_out.view(torch.uint8).cpu().numpy(), plain["q_fp8"])
    assert np.array_equal(w_out.cpu().numpy(), plain["weights"])
    assert np.array_equal(cache.cpu().numpy(), plain["cache"])
    assert np.array_equal(k_cache.cpu().numpy(), plain["cache"])


@pytest.mark.parametrize("n_seq,seq_len,style", [(2, 5120, synth.NEOX), (2, 5120, synth.GPTJ),
                                                  (8, 8192, synth.NEOX)])
def test_k_stream_bulk_and_pdl_modes(n_seq, seq_len, style):
    """The k-only call at prefill size takes the k-stream kernel (more than
    8192 keys): against the oracle on every key, at the bench's 65,536 keys
    too, and with the same bytes under PDL and with its first positions and
    cos/sin rows read before the PDL wait (pdl="early")."""
    inp = synth.make_k_bulk(seed=31, style=style, n_seq=n_seq, seq_len=seq_len,
                            pages=max(200, n_seq * seq_len // 64))
    d = to_device(inp)
    plain = run_k(inp, d)
    assert_parity(inp, plain, run_oracle_k(inp))
    for mode in (True, "early"):
        got = run_k(inp, d, pdl=mode)
        assert np.array_equal(got["cache"], plain["cache"]), mode
    direct = run_k(inp, d, kernel="direct")
    assert np.array_equal(direct["cache"], plain["cache"])


def test_k_stream_error_bits():
    """Bad positions and slots spread over many batches of the k-stream
    kernel's key table: their error bits are set, they write nothing, and
    every other key matches the oracle."""
    inp = synth.make_k_bulk(seed=33, n_seq=2, seq_len=5120, pages=200)
    inp.positions = inp.positions.copy()
    inp.slots = inp.slots.copy()
    inp.positions[[5, 4099]] = [-3, inp.max_position]
    inp.slots[[31, 32, 10239]] = [inp.num_pages * inp.page_size, -1, -64]
    d = to_device(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_k(inp, d, err=err)
    ref = run_oracle_k(inp)
    assert ref["err"] == 3 and int(err.item()) == 3
    assert_parity(inp, got, ref)


def test_head_stride_not_contiguous_uses_per_head_copies():
    """q rows that are not packed head after head (sq_h != 128) take one copy
    per head; the bytes must not change."""
    b = synth.make_decode(seed=17, T=300, H=24, style=synth.NEOX)
    db = to_device(b)
    ref = run_qk(b, db, kernel="pipeline")
    qpad = torch.zeros((300, 24, 136), dtype=torch.bfloat16, device="cuda")
    qpad[:, :, :128] = db["q"]
    dc = dict(db)
    dc["q"] = qpad[:, :, :128]
    got = run_qk(b, dc, kernel="pipeline")
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(got[key], ref[key]), key
    assert_parity(b, got, run_oracle_qk(b))


@pytest.mark.parametrize("page_size", [1, 3, 64])
@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_token_major_cache_layout(page_size, style):
    """The second index-K layout (132 bytes per slot), through both kernels
    and the k-only path; page sizes that are not multiples of 4 are allowed."""
    inp = synth.make_decode(seed=50 + page_size, T=70, H=16, style=style)
    inp.page_size, inp.num_pages = page_size, (4096 * 64) // page_size
    inp.token_major = True
    _check(inp)


def test_token_major_prefill_full_size():
    inp = synth.make_prefill()
    inp.token_major = True
    _check(inp, kernels=("pipeline",))


def test_binding_rejects_host_outputs_and_error_words():
    """A host tensor in an output or error-word slot would hand the kernel a
    host pointer: the binding refuses it before any launch."""
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=15, T=4, H=4)
    d = to_device(inp)
    base = (d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, new_cache(inp), inp.page_size, inp.rope_dim,
            inp.style)
    kw = dict(max_position=inp.max_position)
    with pytest.raises(ValueError):
        dp.dsa_indexer_qk_prepare_store(
            *base, q_fp8_out=torch.empty((4, 4, 128), dtype=torch.uint8), **kw)
    with pytest.raises(ValueError):
        dp.dsa_indexer_qk_prepare_store(
            *base, weights_out=torch.empty((4, 4), dtype=torch.float32), **kw)
    with pytest.raises(TypeError):
        dp.dsa_indexer_qk_prepare_store(
            *base, q_fp8_out=torch.empty((4, 4, 128), dtype=torch.float16, device="cuda"), **kw)
    with pytest.raises(ValueError):
        dp.dsa_indexer_qk_prepare_store(*base, err_flags=torch.zeros(1, dtype=torch.int32), **kw)
    with pytest.raises(ValueError):
        dp.dsa_indexer_k_prepare_store(
            d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
            inp.eps, new_cache(inp).cpu(), inp.page_size, inp.rope_dim, inp.style, **kw)


@pytest.mark.parametrize("kernel", KERNELS)
def test_padded_strides_on_both_kernels(kernel):
    """q with padded head and token strides (the pipeline kernel then copies
    row by row), and cos/sin read from the first rope_dim/2 columns of wider
    tables (cs_stride > rope_dim / 2): the same bytes as contiguous inputs."""
    inp = synth.make_decode(seed=130, T=300, H=24, style=synth.NEOX)
    d = to_device(inp)
    ref = run_qk(inp, d, kernel=kernel)
    qpad = torch.zeros((300, 24, 136), dtype=torch.bfloat16, device="cuda")
    qpad[:, :, :128] = d["q"]
    wide = lambda t: torch.cat([t, torch.full_like(t, 7.0)], dim=1)
    dp_ = dict(d)
    dp_["q"] = qpad[:, :, :128]
    dp_["cos"] = wide(d["cos"])[:, :32]
    dp_["sin"] = wide(d["sin"])[:, :32]
    assert dp_["q"].stride() == (24 * 136, 136, 1) and dp_["cos"].stride(0) == 64
    got = run_qk(inp, dp_, kernel=kernel)
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(got[key], ref[key]), key
    assert_parity(inp, ref, run_oracle_qk(inp))


@pytest.mark.parametrize("H", [32, 16])
def test_prefill_full_size_few_heads(H):
    """Prefill (T = 8192) with 32 and 16 heads: the pipeline kernel packs
    64 / H tokens into a unit (one bulk copy of their query rows)."""
    _check(synth.make_prefill(seed=3 + H, H=H))


@pytest.mark.parametrize("T,H", [(4001, 13), (3901, 24), (4099, 20), (3699, 8)])
def test_multi_token_units_ragged(T, H):
    """Units of several tokens with a ragged last unit, head counts that are
    not a multiple of 4 or 8 (gate weights from global memory), both
    pairings."""
    _check(synth.make_decode(seed=T + H, T=T, H=H, style=(T + H) % 2))


@pytest.mark.parametrize("pad_t,pad_h", [(3, 0), (0, 8)])
def test_multi_token_units_padded_strides(pad_t, pad_h):
    """Units of several tokens whose query rows are not one contiguous block:
    a padded token stride (one bulk copy per token) and a padded head stride
    (one per row); the same bytes as contiguous inputs."""
    T, H = 3700, 16
    inp = synth.make_decode(seed=140 + pad_t, T=T, H=H, style=synth.NEOX)
    d = to_device(inp)
    ref = run_qk(inp, d, kernel="pipeline")
    qpad = torch.zeros((T, H + pad_t, 128 + pad_h), dtype=torch.bfloat16, device="cuda")
    qpad[:, :H, :128] = d["q"]
    dp_ = dict(d)
    dp_["q"] = qpad[:, :H, :128]
    got = run_qk(inp, dp_, kernel="pipeline")
    for key in ("q_fp8", "weights", "cache"):
        assert np.array_equal(got[key], ref[key]), key
    assert_parity(inp, ref, run_oracle_qk(inp))


@pytest.mark.parametrize("T,H", [(3, 1000), (2, 4096)])
def test_many_heads(T, H):
    """Many head chunks per token (the pipeline kernel splits H into chunks
    of at most 64 heads)."""
    _check(synth.make_decode(seed=131 + H, T=T, H=H, style=synth.GPTJ))


@pytest.mark.parametrize("kernel", ["direct", "pipeline"])
def test_prepared_calls_match_binding(kernel):
    """prepare_qk_prepare_store / prepare_k_prepare_store: checked and bound
    once, called twice, they write exactly what the plain binding writes."""
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=91, T=48, H=16)
    d = to_device(inp)
    ref = run_qk(inp, d, kernel=kernel)
    ref_k = run_k(inp, d, kernel=kernel)
    cache = new_cache(inp)
    q_out = torch.empty((inp.T, inp.H, 128), dtype=torch.float8_e4m3fn, device="cuda")
    w_out = torch.empty((inp.T, inp.H), dtype=torch.float32, device="cuda")
    call = dp.prepare_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        q_fp8_out=q_out, weights_out=w_out, max_position=inp.max_position, kernel=kernel)
    for _ in range(2):
        got_q, got_w = call()
        torch.cuda.synchronize()
        assert got_q.data_ptr() == q_out.data_ptr()
        assert np.array_equal(got_q.view(torch.uint8).cpu().numpy(), ref["q_fp8"])
        assert np.array_equal(got_w.cpu().numpy(), ref["weights"])
        assert np.array_equal(cache.cpu().numpy(), ref["cache"])
    cache_k = new_cache(inp)
    kcall = dp.prepare_k_prepare_store(
        d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"], inp.eps,
        cache_k, inp.page_size, inp.rope_dim, inp.style, max_position=inp.max_position,
        kernel=kernel)
    for _ in range(2):
        assert kcall() is None
        torch.cuda.synchronize()
        assert np.array_equal(cache_k.cpu().numpy(), ref_k["cache"])
