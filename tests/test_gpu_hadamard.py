"""The Hadamard-rotated variant (DSA_FLAG_HADAMARD: q heads and k multiplied
by H_128 / sqrt(128) after RoPE) through the C ABI, against the oracle's
Hadamard mode, with the same bar as the plain path: q codes exact (the
butterflies run in the oracle's stage order, so every rounding is shared),
scales and slots exact, k codes within one step in at most 0.1% of elements,
weights within 1e-6.  Both kernels, every rope_dim, both cache layouts, the
error bits, and the full prefill and decode shapes."""
import numpy as np
import pytest
import torch

import synth
from _compare import assert_parity, compare
from _gpu import new_cache, run_k, run_qk, to_device
from _run import run_oracle_qk

pytestmark = pytest.mark.gpu

KERNELS = ("direct", "pipeline")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


def _check(inp, kernels=KERNELS):
    d = to_device(inp)
    ref = run_oracle_qk(inp, hadamard=True)
    first = None
    for kern in kernels:
        gpu = run_qk(inp, d, kernel=kern, hadamard=True)
        rep = assert_parity(inp, gpu, ref)
        gk = run_k(inp, d, kernel=kern, hadamard=True)
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


@pytest.mark.parametrize("rope_dim", [0, 16, 32, 64, 128])
@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_rope_dims(rope_dim, style):
    """Every lane layout: chunks of rope_dim/16 (NeoX), 2*rope_dim/16 (GPT-J)
    or 16 (no RoPE) elements."""
    inp = synth.make_decode(seed=rope_dim + 70, T=40, H=6, style=style)
    inp.cos, inp.sin = synth.rope_table(inp.max_position, max(rope_dim, 16))
    inp.rope_dim = rope_dim
    _check(inp)


def test_decode_gptj():
    _check(synth.make_decode())


@pytest.mark.parametrize("T", [1, 64, 256])
def test_decode_sweep(T):
    _check(synth.make_sweep(T))


def test_prefill_full_size():
    _check(synth.make_prefill(), kernels=("pipeline",))


@pytest.mark.parametrize("T,H", [(3, 5), (33, 13), (517, 100), (5, 128)])
def test_ragged(T, H):
    _check(synth.make_decode(seed=T * 5 + H, T=T, H=H, style=(T + H) % 2))


@pytest.mark.parametrize("page_size", [1, 64])
def test_token_major_cache_layout(page_size):
    inp = synth.make_decode(seed=80 + page_size, T=50, H=8)
    inp.page_size, inp.num_pages = page_size, (4096 * 64) // page_size
    inp.token_major = True
    _check(inp)


def test_device_error_bits():
    inp = synth.make_decode(seed=81, T=20, H=4)
    inp.positions = inp.positions.copy()
    inp.slots = inp.slots.copy()
    inp.positions[3] = -1
    inp.slots[9] = -5
    d = to_device(inp)
    ref = run_oracle_qk(inp, hadamard=True)
    assert ref["err"] == 3
    ok = np.ones(inp.T, bool)
    ok[3] = False
    for kern in KERNELS:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = run_qk(inp, d, err=err, kernel=kern, hadamard=True)
        assert int(err.item()) == 3
        rep = compare(inp, dict(q_fp8=got["q_fp8"][ok], weights=got["weights"][ok],
                                cache=got["cache"]),
                      dict(q_fp8=ref["q_fp8"][ok], weights=ref["weights"][ok], cache=ref["cache"]))
        assert rep["ok"], rep


def test_scores_match_the_plain_path():
    """H_128 / sqrt(128) is orthogonal, so the gated score w'_h (q.k) -- the
    weight carries the q scale 2^e_q -- of the rotated codes equals that of
    the plain codes up to the e4m3 error of both.  Each dequantised element
    is within 2^-4 (relative) of the value it encodes, so each score is
    within about (2 * 2^-4 + 2^-8) |w'| |q| |k| of the exact one
    (Cauchy-Schwarz), and the two within twice that."""
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=82, T=64, H=16)
    d = to_device(inp)
    scores, mass = [], None
    for had in (False, True):
        g = run_qk(inp, d, hadamard=had)
        codes, scales = dp.cache_views(torch.from_numpy(g["cache"]), inp.page_size)
        qd = torch.from_numpy(g["q_fp8"]).view(torch.float8_e4m3fn).double()
        kd = codes[inp.slots].view(torch.float8_e4m3fn).double() * scales[inp.slots, None].double()
        w = g["weights"].astype(np.float64)
        scores.append(w * torch.einsum("thd,td->th", qd, kd).numpy())
        if mass is None:
            mass = np.abs(w) * (qd.norm(dim=2) * kd.norm(dim=1)[:, None]).numpy()
    plain, rot = scores
    bound = 2.0 * (2 * 2.0 ** -4 + 2.0 ** -8) * 1.1 * mass
    assert np.all(np.abs(rot - plain) <= bound)
    assert np.corrcoef(rot.ravel(), plain.ravel())[0, 1] > 0.99


@pytest.mark.parametrize("style", [synth.NEOX, synth.GPTJ])
def test_stress_full_size(style):
    """The heavy-tailed stress set (8 sequences x 8192 tokens, Student-t
    values, all-zero rows, planted near-ties, shuffled pages) at full size."""
    inp = synth.make_stress(style=style)
    _check(inp, kernels=("pipeline",))


@pytest.mark.parametrize("T,H", [(1, 1), (1, 128), (2, 3)])
def test_smallest_shapes(T, H):
    _check(synth.make_decode(seed=100 + T * 7 + H, T=T, H=H, style=(T + H) % 2))


@pytest.mark.parametrize("pdl", [True, "early"])
def test_pdl_graph_of_layers_matches_eager(pdl):
    """Three layers' calls in one CUDA graph with PDL (the second and third
    start while the one before drains): every layer's bytes equal its eager
    call's."""
    import prep_token_gb300 as dp
    layers = [synth.make_decode(seed=110 + i, T=64, H=16) for i in range(3)]
    for inp in layers[1:]:
        inp.positions, inp.slots = layers[0].positions, layers[0].slots
        inp.cos, inp.sin, inp.max_position = layers[0].cos, layers[0].sin, layers[0].max_position
    devs = [to_device(inp) for inp in layers]
    eager = [run_qk(inp, d, hadamard=True) for inp, d in zip(layers, devs)]
    caches = [new_cache(inp) for inp in layers]
    outs = [(torch.empty((64, 16, 128), dtype=torch.float8_e4m3fn, device="cuda"),
             torch.empty((64, 16), dtype=torch.float32, device="cuda")) for _ in layers]

    def call(inp, d, cache, out, s, pdl_mode):
        dp.dsa_indexer_qk_prepare_store(
            d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim,
            inp.style, q_fp8_out=out[0], weights_out=out[1], max_position=inp.max_position,
            pdl=pdl_mode, hadamard=True, stream=s)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for args in zip(layers, devs, caches, outs):
            call(*args, s, False)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for args in zip(layers, devs, caches, outs):
            call(*args, s, pdl)
    for c in caches:
        c.fill_(0xCD)
    g.replay()
    torch.cuda.synchronize()
    for e, c, (qo, wo) in zip(eager, caches, outs):
        assert np.array_equal(qo.view(torch.uint8).cpu().numpy(), e["q_fp8"])
        assert np.array_equal(wo.cpu().numpy(), e["weights"])
        assert np.array_equal(c.cpu().numpy(), e["cache"])


@pytest.mark.parametrize("T,H", [(4001, 16), (3901, 24)])
def test_multi_token_units(T, H):
    """The Hadamard variant on units of several tokens (pipeline kernel)."""
    _check(synth.make_decode(seed=T + H + 7, T=T, H=H, style=(T + H) % 2))
