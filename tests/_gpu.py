"""GPU-side test helpers: move a synth.Inputs to the device, call the C ABI
through the binding, bring the outputs back as numpy."""
import numpy as np
import torch

import prep_token_gb300 as dp

SENTINEL = 0xCD


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(inp, device="cuda"):
    d = {}
    d["q"] = bf16_tensor(inp.q, device)
    if inp.kw is not None:
        kw = bf16_tensor(inp.kw, device)
        d["kw"] = kw
        d["k"], d["w"] = kw[:, :128], kw[:, 128:128 + inp.H]
    else:
        d["k"], d["w"] = bf16_tensor(inp.k, device), bf16_tensor(inp.w, device)
    d["positions"] = torch.from_numpy(inp.positions).to(device)
    d["slots"] = torch.from_numpy(inp.slots).to(device)
    d["cos"] = torch.from_numpy(inp.cos).to(device)
    d["sin"] = torch.from_numpy(inp.sin).to(device)
    d["gamma"] = torch.from_numpy(inp.gamma).to(device)
    d["beta"] = torch.from_numpy(inp.beta).to(device)
    return d


def new_cache(inp, device="cuda", fill=SENTINEL):
    return torch.full((inp.cache_bytes,), fill, dtype=torch.uint8, device=device)


def _layout_kw(inp, kw):
    kw.setdefault("cache_layout", "token_major" if inp.token_major else "paged")
    return kw


def run_qk(inp, d, cache=None, err=None, **kw):
    kw = _layout_kw(inp, kw)
    cache = new_cache(inp) if cache is None else cache
    q_fp8, weights = dp.dsa_indexer_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, cache, inp.page_size, inp.rope_dim, inp.style,
        err_flags=err, max_position=inp.max_position, **kw)
    torch.cuda.synchronize()
    return dict(q_fp8=q_fp8.view(torch.uint8).cpu().numpy(), weights=weights.cpu().numpy(),
                cache=cache.cpu().numpy())


def run_k(inp, d, cache=None, err=None, **kw):
    kw = _layout_kw(inp, kw)
    cache = new_cache(inp) if cache is None else cache
    dp.dsa_indexer_k_prepare_store(
        d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"], inp.eps,
        cache, inp.page_size, inp.rope_dim, inp.style, err_flags=err,
        max_position=inp.max_position, **kw)
    torch.cuda.synchronize()
    return dict(cache=cache.cpu().numpy())
