"""The C ABI without a GPU: the library builds and loads, exports every
function include/dsa_prep.h declares, and rejects bad arguments on the host
before any CUDA call (these calls never reach a launch)."""
import ctypes
import os
import re

import pytest

import prep_token_gb300 as dp
from prep_token_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return dp.library()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[\w\s\*]*?\b(dsa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"dsa_indexer_qk_prepare_store", "dsa_indexer_k_prepare_store",
            "dsa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(6):
        assert dp.dsa_status_string(s)
    assert lib.dsa_prep_version() >> 16 == 3


A = 0x10000  # a 16-byte aligned fake address: only used by calls that must fail validation


def _qk(lib, **over):
    args = dict(q=A, sqt=64 * 128, sqh=128, k=A, skt=128, w=A, swt=64, pos=A, loc=A, cos=A,
                sin=A, cs=32, maxpos=4096, g=A, b=A, eps=1e-6, sm=0.088, qo=A, wo=A, cache=A,
                pages=4, ps=64, T=4, H=64, D=128, r=64, style=0, flags=0, err=None, stream=None)
    args.update(over)
    return lib.dsa_indexer_qk_prepare_store(*args.values())


def _k(lib, **over):
    args = dict(k=A, skt=128, pos=A, loc=A, cos=A, sin=A, cs=32, maxpos=4096, g=A, b=A,
                eps=1e-6, cache=A, pages=4, ps=64, T=4, D=128, r=64, style=0, flags=0, err=None,
                stream=None)
    args.update(over)
    return lib.dsa_indexer_k_prepare_store(*args.values())


@pytest.mark.parametrize("over,status", [
    (dict(T=-1), 3), (dict(D=64), 4), (dict(r=8), 4), (dict(r=144), 4), (dict(style=2), 4),
    (dict(eps=float("nan")), 4), (dict(ps=0), 3), (dict(pages=0), 3), (dict(maxpos=0), 3),
    (dict(k=None), 1), (dict(pos=None), 1), (dict(cache=None), 1), (dict(cos=None), 1),
    (dict(ps=6), 2), (dict(k=A + 8), 2), (dict(skt=132), 2), (dict(pos=A + 4), 2),
    (dict(g=A + 4), 2), (dict(cache=A + 8), 2), (dict(cos=A + 4), 2), (dict(cs=34), 2),
    (dict(cs=16), 3), (dict(skt=-128), 3), (dict(flags=64), 4), (dict(flags=6), 4), (dict(flags=8), 4),
    (dict(flags=32 | 8), 4), (dict(flags=32 | 6), 4), (dict(flags=0x80000000), 4),
    (dict(flags=1 << 30), 4), (dict(flags=(1 << 30) | 4), 4),
    (dict(r=48), 4), (dict(r=96), 4), (dict(r=112), 4),
])
def test_k_side_validation(lib, over, status):
    assert _k(lib, **over) == status
    assert _qk(lib, **over) == status


@pytest.mark.parametrize("over,status", [
    (dict(H=0), 3), (dict(H=5000), 3), (dict(swt=32), 3), (dict(sqt=-1), 3),
    (dict(q=None), 1), (dict(w=None), 1), (dict(qo=None), 1), (dict(wo=None), 1),
    (dict(q=A + 2), 2), (dict(sqt=64 * 128 + 4), 2), (dict(sqh=132), 2), (dict(w=A + 1), 2),
    (dict(qo=A + 8), 2), (dict(wo=A + 2), 2), (dict(sm=float("inf")), 4),
])
def test_q_side_validation(lib, over, status):
    assert _qk(lib, **over) == status


def test_empty_batch_is_ok_without_pointers(lib):
    nulls = dict(q=None, k=None, w=None, pos=None, loc=None, cos=None, sin=None, g=None,
                 b=None, qo=None, wo=None, cache=None)
    assert _qk(lib, T=0, **nulls) == 0
    assert _k(lib, T=0, **{k: v for k, v in nulls.items() if k in
                           ("k", "pos", "loc", "cos", "sin", "g", "b", "cache")}) == 0


def test_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        dp.dsa_indexer_qk_prepare_store(q, q[:, 0], q[:, :, 0], None, None, None, None, None,
                                        None, 1e-6, 0.1, None, 64)


def _unf(lib, **over):
    args = dict(q=A, sqt=64 * 128, sqh=128, k=A, skt=128, w=A, swt=64, pos=A, loc=A, cos=A,
                sin=A, cs=32, maxpos=4096, g=A, b=A, eps=1e-6, sm=0.088, qo=A, wo=A, cache=A,
                pages=4, ps=64, T=4, H=64, D=128, r=64, style=0, flags=0, ws=0x100000,
                wsb=1 << 20, err=None, stream=None)
    args.update(over)
    return lib.dsa_indexer_qk_prepare_store_unfused(*args.values())


def test_unfused_workspace_size(lib):
    assert lib.dsa_unfused_workspace_bytes(4, 64) == 2 * 1024 + 4 * 64 * 256
    assert lib.dsa_unfused_workspace_bytes(3, 5) == 2 * 768 + 3 * 5 * 256
    assert lib.dsa_unfused_workspace_bytes(-1, 5) == 0
    assert lib.dsa_unfused_workspace_bytes(4, 0) == 0


@pytest.mark.parametrize("over,status", [
    (dict(T=-1), 3), (dict(H=0), 3), (dict(D=64), 4), (dict(r=48), 4), (dict(style=3), 4),
    (dict(flags=2), 4), (dict(flags=32), 4), (dict(ws=None), 1), (dict(wsb=1000), 3), (dict(ws=0x100000 + 16), 2),
    (dict(q=A + 2), 2), (dict(cache=None), 1), (dict(ps=6), 2), (dict(swt=8), 3),
])
def test_unfused_validation(lib, over, status):
    assert _unf(lib, **over) == status


def test_unfused_empty_batch(lib):
    assert _unf(lib, T=0, q=None, k=None, ws=None, wsb=0) == 0


def _lg(lib, **over):
    args = dict(q=A, w=A, cache=A, pages=4, ps=64, bt=A, bts=4, lens=A, out=A, outs=128,
                maxc=128, T=2, H=64, flags=0, err=None, stream=None)
    args.update(over)
    return lib.dsa_indexer_mqa_logits(*args.values())


@pytest.mark.parametrize("over,status", [
    (dict(T=-1), 3), (dict(T=70000), 3), (dict(H=48), 4), (dict(ps=32), 4), (dict(pages=0), 3),
    (dict(bts=-1), 3), (dict(outs=64), 3), (dict(flags=2), 4), (dict(flags=128), 4),
    (dict(flags=64), 4),  # DSA_FLAG_PDL_EARLY_INDEX needs DSA_FLAG_PDL
    (dict(q=None), 1), (dict(lens=None), 1), (dict(q=A + 8), 2), (dict(cache=A + 4), 2),
    (dict(w=A + 2), 2),
    (dict(bts=1), 3), (dict(maxc=257, outs=300, bts=4), 3),  # rows must cover max_context
])
def test_logits_validation(lib, over, status):
    assert _lg(lib, **over) == status


def test_logits_empty_batch_is_ok_without_pointers(lib):
    assert _lg(lib, T=0, q=None, w=None, bt=None, lens=None, out=None) == 0
