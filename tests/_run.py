"""Test helpers: run the oracle on a synth.Inputs, compare E4M3 code arrays."""
import numpy as np

import oracle

SENTINEL = 0xCD


def code_ordinal(c):
    """E4M3 code -> signed position on the number line (+0 and -0 equal)."""
    c = np.asarray(c, np.uint8).astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def code_distance(a, b):
    return np.abs(code_ordinal(a) - code_ordinal(b))


def fresh_cache(inp, fill=SENTINEL):
    return np.full(inp.cache_bytes, fill, np.uint8)


def run_oracle_qk(inp, cache=None, T=None, chain=False, hadamard=False):
    T = inp.T if T is None else T
    cache = fresh_cache(inp) if cache is None else cache
    q_fp8 = np.zeros((max(T, 1), inp.H, 128), np.uint8)
    weights = np.zeros((max(T, 1), inp.H), np.float32)
    w_buf = inp.kw if inp.kw is not None else inp.w
    # w's row stride refers to the buffer; pass a flat view that starts at w[0, 0]
    w_flat = w_buf.reshape(-1)[128:] if inp.kw is not None else w_buf.reshape(-1)
    err, qe, ke = oracle.qk_prepare_store(
        inp.q.reshape(-1), inp.q_stride_t, inp.q_stride_h,
        inp.k_buffer().reshape(-1), inp.k_stride_t,
        np.ascontiguousarray(w_flat), inp.w_stride_t,
        inp.positions[:T], inp.slots[:T], inp.cos, inp.sin, inp.cs_stride,
        inp.max_position, inp.gamma, inp.beta, inp.eps, inp.softmax_scale,
        q_fp8, weights, cache, inp.num_pages, inp.page_size, inp.H, inp.rope_dim,
        inp.style, T=T, chain=chain, token_major=inp.token_major, hadamard=hadamard)
    return dict(q_fp8=q_fp8[:T], weights=weights[:T], cache=cache, err=err,
                q_exp=qe, k_exp=ke)


def run_oracle_k(inp, cache=None, bf16_intermediate=False, T=None):
    T = inp.T if T is None else T
    cache = fresh_cache(inp) if cache is None else cache
    err, ke = oracle.k_prepare_store(
        inp.k_buffer().reshape(-1), inp.k_stride_t, inp.positions[:T], inp.slots[:T],
        inp.cos, inp.sin, inp.cs_stride, inp.max_position, inp.gamma, inp.beta,
        inp.eps, cache, inp.num_pages, inp.page_size, inp.rope_dim, inp.style,
        bf16_intermediate=bf16_intermediate, T=T, token_major=inp.token_major)
    return dict(cache=cache, err=err, k_exp=ke)


def cache_views(inp, cache):
    """(codes[num_pages*page_size, 128], scales[num_pages*page_size]) of the
    index-K cache: page-blocked (page p = [page_size x 128 codes][page_size x
    fp32]) or token-major (132 bytes per slot)."""
    if inp.token_major:
        rows = cache.reshape(-1, 132)
        return rows[:, :128], np.ascontiguousarray(rows[:, 128:]).view(np.float32).reshape(-1)
    P = inp.page_size
    pages = cache.reshape(inp.num_pages, P * 132)
    codes = pages[:, :P * 128].reshape(inp.num_pages * P, 128)
    scales = np.ascontiguousarray(pages[:, P * 128:]).view(np.float32).reshape(-1)
    return codes, scales
