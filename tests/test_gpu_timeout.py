"""The pipeline kernel's bounded waits, exercised without a fault.

DSA_FLAG_TEST_WITHHOLD_UNIT makes the first CTA's producer never fill its
first ring stage.  The consumers' waits on it give up after their 2 s limit,
the CTA stops and reports DSA_DEVERR_TIMEOUT, every other CTA completes, and
the context stays usable: a normal call right after it still matches the
oracle."""
import time

import numpy as np
import pytest
import torch

import synth
from _compare import assert_parity
from _gpu import new_cache, run_qk, to_device
from _run import run_oracle_qk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prep_token_gb300 as dp
    dp.library()


def test_withheld_stage_times_out_and_context_survives():
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=90, T=512, H=64)
    d = to_device(inp)
    cache = new_cache(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args, outs, _, _ = dp._qk_args(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        None, None, None, inp.max_position)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = dp.library().dsa_indexer_qk_prepare_store(
        *args, dp.FLAG_PIPELINE | dp.FLAG_TEST_WITHHOLD_UNIT, err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) & dp.DEVERR_TIMEOUT
    assert 1.5 < dt < 30.0, dt
    # the context is intact: the same call without the hook is exact again
    err.zero_()
    got = run_qk(inp, d, err=err, kernel="pipeline")
    assert int(err.item()) == 0
    assert_parity(inp, got, run_oracle_qk(inp))


def test_hook_requires_the_pipeline_kernel():
    import prep_token_gb300 as dp
    inp = synth.make_decode(seed=91, T=8, H=4)
    d = to_device(inp)
    args, _, _, _ = dp._qk_args(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, new_cache(inp), inp.page_size, inp.rope_dim,
        inp.style, None, None, None, inp.max_position)
    st = dp.library().dsa_indexer_qk_prepare_store(
        *args, dp.FLAG_TEST_WITHHOLD_UNIT, None, torch.cuda.current_stream().cuda_stream)
    assert st == 4  # DSA_ERR_UNSUPPORTED, nothing launched
