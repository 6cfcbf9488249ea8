"""DSA indexer Q/K prepare-and-store on GB300 (sm_103a).

A thin Python binding over the C ABI of ``libdsaprep.so`` (declared in
``include/dsa_prep.h``): it checks tensor dtypes and devices, allocates the
outputs the caller did not pass, and forwards data pointers, strides and the
current CUDA stream.  Every step of the path runs in the library's kernels;
there is no CPU or PyTorch fallback, and a missing library raises.

What the calls compute follows the sglang PR "[AMD] [GLM5] Fuse the DSA
indexer Q/K rope + quant + K-cache write" (Motivation, Modifications) and the
vllm PR "[ROCm][Perf] Enable fused indexer-Q RoPE+quant kernel for
DeepSeek/GLM sparse attention" (Summary): RoPE on q and k, LayerNorm on k,
e4m3 quantisation with one power-of-two scale per 128 values, the gate-weight
fold, and the paged index-K cache write.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from ._build import LIB_PATH

__all__ = [
    "DsaError", "NEOX", "GPTJ", "HEAD_DIM", "DEVERR_POSITION", "DEVERR_SLOT", "DEVERR_TIMEOUT",
    "DEVERR_INTERNAL",
    "FLAG_PDL", "FLAG_PIPELINE", "FLAG_DIRECT", "FLAG_PDL_EARLY_ROPE", "FLAG_CACHE_TOKEN_MAJOR",
    "FLAG_HADAMARD", "FLAG_PDL_EARLY_INDEX",
    "dsa_indexer_qk_prepare_store", "dsa_indexer_k_prepare_store", "dsa_status_string",
    "dsa_indexer_qk_prepare_store_unfused", "dsa_unfused_workspace_bytes",
    "dsa_indexer_qk_prepare_store_unfused_noalloc", "dsa_indexer_mqa_logits",
    "library", "cache_bytes", "cache_views",
    "PreparedCall", "prepare_qk_prepare_store", "prepare_k_prepare_store",
]

NEOX, GPTJ = 0, 1
HEAD_DIM = 128
DEVERR_POSITION, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_INTERNAL = 1, 2, 4, 8
FLAG_PDL, FLAG_PIPELINE, FLAG_DIRECT, FLAG_PDL_EARLY_ROPE = 1, 2, 4, 8
FLAG_CACHE_TOKEN_MAJOR = 16
FLAG_HADAMARD = 32
FLAG_PDL_EARLY_INDEX = 64
FLAG_TEST_WITHHOLD_UNIT = 1 << 30  # test only: see include/dsa_prep.h
_LAYOUT_FLAGS = {"paged": 0, "token_major": FLAG_CACHE_TOKEN_MAJOR}
_KERNEL_FLAGS = {"auto": 0, "pipeline": FLAG_PIPELINE, "direct": FLAG_DIRECT}
ROW_BYTES = HEAD_DIM + 4  # 128 codes + one fp32 scale per slot

_STATUS = {0: "DSA_OK", 1: "DSA_ERR_NULL", 2: "DSA_ERR_ALIGN", 3: "DSA_ERR_SHAPE",
           4: "DSA_ERR_UNSUPPORTED", 5: "DSA_ERR_LAUNCH", 6: "DSA_ERR_SCRATCH_LIMIT"}


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)} ({dsa_status_string(status)})")


_lib = None


def library() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'); there is no fallback implementation")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        U32 = ctypes.c_uint32
        lib.dsa_indexer_qk_prepare_store.argtypes = [
            P, I64, I64, P, I64, P, I64, P, P, P, P, I64, I64, P, P, F32, F32, P, P, P, I64, I32,
            I32, I32, I32, I32, I32, U32, P, P]
        lib.dsa_indexer_qk_prepare_store.restype = ctypes.c_int
        lib.dsa_indexer_k_prepare_store.argtypes = [
            P, I64, P, P, P, P, I64, I64, P, P, F32, P, I64, I32, I32, I32, I32, I32, U32, P, P]
        lib.dsa_indexer_k_prepare_store.restype = ctypes.c_int
        SZ = ctypes.c_size_t
        lib.dsa_unfused_workspace_bytes.argtypes = [I32, I32]
        lib.dsa_unfused_workspace_bytes.restype = SZ
        lib.dsa_indexer_qk_prepare_store_unfused.argtypes = [
            P, I64, I64, P, I64, P, I64, P, P, P, P, I64, I64, P, P, F32, F32, P, P, P, I64, I32,
            I32, I32, I32, I32, I32, U32, P, SZ, P, P]
        lib.dsa_indexer_qk_prepare_store_unfused.restype = ctypes.c_int
        lib.dsa_indexer_qk_prepare_store_unfused_noalloc.argtypes = [
            P, I64, I64, P, I64, P, I64, P, P, P, P, I64, I64, P, P, F32, F32, P, P, P, I64, I32,
            I32, I32, I32, I32, I32, U32, P, P]
        lib.dsa_indexer_qk_prepare_store_unfused_noalloc.restype = ctypes.c_int
        lib.dsa_indexer_mqa_logits.argtypes = [
            P, P, P, I64, I32, P, I64, P, P, I64, I32, I32, I32, U32, P, P]
        lib.dsa_indexer_mqa_logits.restype = ctypes.c_int
        lib.dsa_status_string.argtypes = [ctypes.c_int]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_prep_version.argtypes = []
        lib.dsa_prep_version.restype = ctypes.c_int32
        _lib = lib
    return _lib


def dsa_status_string(status: int) -> str:
    return library().dsa_status_string(status).decode()


def cache_bytes(num_pages: int, page_size: int) -> int:
    return num_pages * page_size * ROW_BYTES


def cache_views(index_k_cache: torch.Tensor, page_size: int):
    """(codes [slots, 128] uint8, scales [slots] fp32) views of a paged
    index-K cache: page p = [page_size x 128 codes][page_size x fp32 scale]."""
    flat = index_k_cache.reshape(-1).view(torch.uint8)
    num_pages = flat.numel() // (page_size * ROW_BYTES)
    pages = flat[: num_pages * page_size * ROW_BYTES].view(num_pages, page_size * ROW_BYTES)
    codes = pages[:, : page_size * HEAD_DIM].reshape(num_pages * page_size, HEAD_DIM)
    scales = pages[:, page_size * HEAD_DIM:].contiguous().view(torch.float32).reshape(-1)
    return codes, scales


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, dim: int | None = None, device=None):
    """dtype (one torch dtype or a tuple of them), rank, a CUDA device (the
    given one when `device` is set) and a contiguous innermost dimension."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device (no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other tensors on {device}")
    if t.dtype is not dtype and not (isinstance(dtype, tuple) and t.dtype in dtype):
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    nd = t.dim()
    if dim is not None and nd != dim:
        raise ValueError(f"{name}: expected {dim} dims, got {tuple(t.shape)}")
    if nd and t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"{name}: innermost dimension must be contiguous")


def _num_pages(index_k_cache: torch.Tensor, page_size: int) -> int:
    if not index_k_cache.is_contiguous():
        raise ValueError("index_k_cache must be contiguous")
    nbytes = index_k_cache.numel() * index_k_cache.element_size()
    if page_size < 1 or nbytes % (page_size * ROW_BYTES):
        raise ValueError("index_k_cache size is not a whole number of pages")
    return nbytes // (page_size * ROW_BYTES)


def _layout(cache_layout: str) -> int:
    if cache_layout not in _LAYOUT_FLAGS:
        raise ValueError(f"cache_layout must be one of {sorted(_LAYOUT_FLAGS)}")
    return _LAYOUT_FLAGS[cache_layout]


def _flags(pdl, kernel: str) -> int:
    """pdl: False, True, or "early" (PDL plus FLAG_PDL_EARLY_ROPE: positions,
    slots and the cos/sin cache are not written by the previous kernel)."""
    if kernel not in _KERNEL_FLAGS:
        raise ValueError(f"kernel must be one of {sorted(_KERNEL_FLAGS)}")
    if pdl not in (False, True, "early"):
        raise ValueError('pdl must be False, True or "early"')
    f = FLAG_PDL if pdl else 0
    if pdl == "early":
        f |= FLAG_PDL_EARLY_ROPE
    return f | _KERNEL_FLAGS[kernel]


def _err_ptr(err_flags, device):
    """The device error word: an int32 CUDA tensor on the call's device."""
    if err_flags is None:
        return None
    _need(err_flags, "err_flags", torch.int32, None, device)
    if err_flags.numel() < 1:
        raise ValueError("err_flags must hold at least one int32")
    return err_flags.data_ptr()


def _on(device):
    """The tensors' device made current for a library call (the C side takes
    the SM count, kernel attributes and scratch address from the current
    device); a no-op when it already is."""
    if device.index is None or torch.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream(stream, device=None) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _k_common(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta,
              index_k_cache, rope_dim):
    _need(k, "k", torch.bfloat16, 2)
    dev = k.device
    _need(positions, "positions", torch.int64, 1, dev)
    _need(out_cache_loc, "out_cache_loc", torch.int64, 1, dev)
    _need(ln_gamma, "ln_gamma", torch.float32, 1, dev)
    _need(ln_beta, "ln_beta", torch.float32, 1, dev)
    if not isinstance(index_k_cache, torch.Tensor) or index_k_cache.device != dev:
        raise ValueError(f"index_k_cache must be a tensor on {dev}")
    if rope_dim:
        _need(cos_cache, "cos_cache", torch.float32, 2, dev)
        _need(sin_cache, "sin_cache", torch.float32, 2, dev)
        if cos_cache.stride(0) != sin_cache.stride(0) or cos_cache.shape[0] != sin_cache.shape[0]:
            raise ValueError("cos_cache and sin_cache must share rows and row stride")
        return cos_cache.stride(0), cos_cache.shape[0]
    return 0, 1 << 62


def _qk_args(q, k, w, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta,
             ln_eps, softmax_scale, index_k_cache, page_size, rope_dim, rope_style, q_fp8_out,
             weights_out, num_tokens, max_position):
    """Checks and the C argument list shared by the fused and unfused calls,
    up to and including rope_style; also returns the two outputs."""
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    _need(w, "w", torch.bfloat16, 2, dev)
    cs_stride, rows = _k_common(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma,
                                ln_beta, index_k_cache, rope_dim)
    if k.device != dev:
        raise ValueError(f"k is on {k.device}, q on {dev}")
    T = q.shape[0] if num_tokens is None else int(num_tokens)
    H = q.shape[1]
    if q.shape[2] != HEAD_DIM:
        raise ValueError("q: head_dim must be 128")
    for name, t in (("k", k), ("w", w), ("positions", positions), ("out_cache_loc", out_cache_loc)):
        if t.shape[0] < T:
            raise ValueError(f"{name} has fewer than {T} rows")
    if w.shape[1] != H:
        raise ValueError("w must be [T, H]")
    if q_fp8_out is None:
        q_fp8_out = torch.empty((T, H, HEAD_DIM), dtype=torch.float8_e4m3fn, device=dev)
    if weights_out is None:
        weights_out = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(q_fp8_out, "q_fp8_out", (torch.float8_e4m3fn, torch.uint8), None, dev)
    _need(weights_out, "weights_out", torch.float32, None, dev)
    if q_fp8_out.numel() < T * H * HEAD_DIM or not q_fp8_out.is_contiguous():
        raise ValueError("q_fp8_out must be contiguous [T, H, 128]")
    if not weights_out.is_contiguous() or weights_out.numel() < T * H:
        raise ValueError("weights_out must be contiguous fp32 [T, H]")
    max_position = rows if max_position is None else int(max_position)
    args = (_ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), _ptr(w), w.stride(0),
            _ptr(positions), _ptr(out_cache_loc), _ptr(cos_cache) if rope_dim else None,
            _ptr(sin_cache) if rope_dim else None, cs_stride, max_position, _ptr(ln_gamma),
            _ptr(ln_beta), float(ln_eps), float(softmax_scale), _ptr(q_fp8_out),
            _ptr(weights_out), _ptr(index_k_cache), _num_pages(index_k_cache, page_size),
            page_size, T, H, HEAD_DIM, rope_dim, int(rope_style))
    outs = (q_fp8_out[:T] if q_fp8_out.dim() == 3 and q_fp8_out.shape[0] != T else q_fp8_out,
            weights_out[:T] if weights_out.dim() == 2 and weights_out.shape[0] != T
            else weights_out)
    return args, outs, T, H


def dsa_indexer_qk_prepare_store(q, k, w, positions, out_cache_loc, cos_cache, sin_cache,
                                 ln_gamma, ln_beta, ln_eps, softmax_scale, index_k_cache,
                                 page_size, rope_dim=64, rope_style=NEOX, *, q_fp8_out=None,
                                 weights_out=None, err_flags=None, num_tokens=None,
                                 max_position=None, pdl=False, kernel="auto",
                                 cache_layout="paged", hadamard=False, stream=None):
    """Fused Q/K prepare-and-store (one kernel launch).

    q [T, H, 128] bf16, k [T, 128] bf16, w [T, H] bf16 (row strides of any
    view are honoured), positions/out_cache_loc [T] int64, cos/sin caches
    [max_position, >= rope_dim/2] fp32, ln_gamma/ln_beta [128] fp32,
    index_k_cache: a contiguous CUDA buffer of whole pages (written in place).
    ``num_tokens`` limits the call to the first T live tokens (the graph
    split-op contract); outputs are sized to it.  ``pdl`` launches with
    programmatic dependent launch (the kernel may start while the previous
    kernel of the stream drains; it still waits for that kernel's memory);
    ``pdl="early"`` also reads positions, slots and cos/sin before that wait
    (only when the previous kernel does not write them).
    ``kernel`` = "auto" | "direct" | "pipeline" overrides the size-based
    choice between the two kernels (same bytes either way).
    ``cache_layout`` = "paged" (a page's codes, then its scales) or
    "token_major" (132 bytes per slot: codes, then scale).
    ``hadamard=True`` rotates every q head and k by H_128 / sqrt(128) after
    RoPE, before they are quantised.
    Returns (q_fp8 [T, H, 128] float8_e4m3fn, weights [T, H] fp32)."""
    args, outs, _, _ = _qk_args(q, k, w, positions, out_cache_loc, cos_cache, sin_cache,
                                ln_gamma, ln_beta, ln_eps, softmax_scale, index_k_cache,
                                page_size, rope_dim, rope_style, q_fp8_out, weights_out,
                                num_tokens, max_position)
    with _on(q.device):
        st = library().dsa_indexer_qk_prepare_store(
            *args, _flags(pdl, kernel) | _layout(cache_layout) | (FLAG_HADAMARD if hadamard else 0),
            _err_ptr(err_flags, q.device), _stream(stream, q.device))
    if st != 0:
        raise DsaError(st, "dsa_indexer_qk_prepare_store")
    return outs


def dsa_unfused_workspace_bytes(T: int, H: int) -> int:
    """Workspace the unfused chain needs (bf16 intermediates)."""
    return int(library().dsa_unfused_workspace_bytes(int(T), int(H)))


def dsa_indexer_qk_prepare_store_unfused(q, k, w, positions, out_cache_loc, cos_cache,
                                         sin_cache, ln_gamma, ln_beta, ln_eps, softmax_scale,
                                         index_k_cache, page_size, rope_dim=64,
                                         rope_style=NEOX, *, q_fp8_out=None, weights_out=None,
                                         workspace=None, err_flags=None, num_tokens=None,
                                         max_position=None, pdl=False, cache_layout="paged",
                                         stream=None):
    """The same computation as four launches (LayerNorm, RoPE, q quant + fold,
    k quant + store) with bf16 intermediates in ``workspace`` (a CUDA uint8
    tensor of at least dsa_unfused_workspace_bytes(T, H) bytes; allocated here
    when not given).  The baseline the fused call is measured against."""
    args, outs, T, H = _qk_args(q, k, w, positions, out_cache_loc, cos_cache, sin_cache,
                                ln_gamma, ln_beta, ln_eps, softmax_scale, index_k_cache,
                                page_size, rope_dim, rope_style, q_fp8_out, weights_out,
                                num_tokens, max_position)
    need = dsa_unfused_workspace_bytes(T, H)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if not isinstance(workspace, torch.Tensor) or workspace.device != q.device \
            or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {q.device}")
    nbytes = workspace.numel() * workspace.element_size()
    with _on(q.device):
        st = library().dsa_indexer_qk_prepare_store_unfused(
            *args, (FLAG_PDL if pdl else 0) | _layout(cache_layout), _ptr(workspace), nbytes,
            _err_ptr(err_flags, q.device), _stream(stream, q.device))
    if st != 0:
        raise DsaError(st, "dsa_indexer_qk_prepare_store_unfused")
    return outs


def dsa_indexer_qk_prepare_store_unfused_noalloc(q, k, w, positions, out_cache_loc, cos_cache,
                                                 sin_cache, ln_gamma, ln_beta, ln_eps,
                                                 softmax_scale, index_k_cache, page_size,
                                                 rope_dim=64, rope_style=NEOX, *, q_fp8_out,
                                                 weights_out, err_flags=None, num_tokens=None,
                                                 max_position=None, pdl=False,
                                                 cache_layout="paged", stream=None):
    """The unfused chain with its intermediates in the library's own 32 MiB
    device buffer, for callers that cannot allocate device memory when they
    run it (an engine whose memory pool owns the whole GPU, a plugin handed
    only input and output pointers).  Nothing is allocated here either: the
    caller passes q_fp8_out and weights_out.  Calls that overlap on the GPU
    share the buffer and race; calls with T * (H + 2) * 256 bytes of
    intermediates above 32 MiB raise DsaError (DSA_ERR_SCRATCH_LIMIT)."""
    if q_fp8_out is None or weights_out is None:
        raise ValueError("pass q_fp8_out and weights_out: this entry point allocates nothing")
    args, outs, _, _ = _qk_args(q, k, w, positions, out_cache_loc, cos_cache, sin_cache,
                                ln_gamma, ln_beta, ln_eps, softmax_scale, index_k_cache,
                                page_size, rope_dim, rope_style, q_fp8_out, weights_out,
                                num_tokens, max_position)
    with _on(q.device):
        st = library().dsa_indexer_qk_prepare_store_unfused_noalloc(
            *args, (FLAG_PDL if pdl else 0) | _layout(cache_layout), _err_ptr(err_flags, q.device),
            _stream(stream, q.device))
    if st != 0:
        raise DsaError(st, "dsa_indexer_qk_prepare_store_unfused_noalloc")
    return outs


def _k_args(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta, ln_eps,
            index_k_cache, page_size, rope_dim, rope_style, num_tokens, max_position):
    """Checks and the C argument list of the k-only call, up to rope_style."""
    cs_stride, rows = _k_common(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma,
                                ln_beta, index_k_cache, rope_dim)
    T = k.shape[0] if num_tokens is None else int(num_tokens)
    if k.shape[1] != HEAD_DIM:
        raise ValueError("k: head_dim must be 128")
    for name, t in (("positions", positions), ("out_cache_loc", out_cache_loc)):
        if t.shape[0] < T:
            raise ValueError(f"{name} has fewer than {T} rows")
    max_position = rows if max_position is None else int(max_position)
    return (_ptr(k), k.stride(0), _ptr(positions), _ptr(out_cache_loc),
            _ptr(cos_cache) if rope_dim else None, _ptr(sin_cache) if rope_dim else None,
            cs_stride, max_position, _ptr(ln_gamma), _ptr(ln_beta), float(ln_eps),
            _ptr(index_k_cache), _num_pages(index_k_cache, page_size), page_size, T, HEAD_DIM,
            rope_dim, int(rope_style))


def dsa_indexer_k_prepare_store(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma,
                                ln_beta, ln_eps, index_k_cache, page_size, rope_dim=64,
                                rope_style=NEOX, *, err_flags=None, num_tokens=None,
                                max_position=None, pdl=False, kernel="auto",
                                cache_layout="paged", hadamard=False, stream=None):
    """k-only prepare-and-store (one kernel launch); writes the cache in place.
    ``hadamard=True`` rotates k by H_128 / sqrt(128) after RoPE."""
    args = _k_args(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta, ln_eps,
                   index_k_cache, page_size, rope_dim, rope_style, num_tokens, max_position)
    with _on(k.device):
        st = library().dsa_indexer_k_prepare_store(
            *args, _flags(pdl, kernel) | _layout(cache_layout) | (FLAG_HADAMARD if hadamard else 0),
            _err_ptr(err_flags, k.device), _stream(stream, k.device))
    if st != 0:
        raise DsaError(st, "dsa_indexer_k_prepare_store")


class PreparedCall:
    """One library call whose arguments were checked and converted once.

    For callers with fixed buffers (static activation buffers, or the tensors
    a CUDA graph was captured on): the checks of the plain binding cost about
    ten microseconds of host time per call, while a prepared call is a single
    ctypes call with pre-built arguments.  The tensors it was prepared on must
    stay alive and in place, the stream is the one given (or current) at
    preparation, and the call raises DsaError on a non-zero status.  Calling
    it returns the outputs it writes (for the fused call: q_fp8, weights)."""

    def __init__(self, fn, name, args, device, outs=None, keep=()):
        self._fn = fn
        self._name = name
        self._device = device
        self._args = tuple(t(a) if a is not None else None for t, a in zip(fn.argtypes, args))
        self._outs = outs
        self._keep = keep  # tensors whose pointers the arguments hold

    def __call__(self):
        with _on(self._device):
            st = self._fn(*self._args)
        if st != 0:
            raise DsaError(st, self._name)
        return self._outs


def prepare_qk_prepare_store(q, k, w, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma,
                             ln_beta, ln_eps, softmax_scale, index_k_cache, page_size,
                             rope_dim=64, rope_style=NEOX, *, q_fp8_out=None, weights_out=None,
                             err_flags=None, num_tokens=None, max_position=None, pdl=False,
                             kernel="auto", cache_layout="paged", hadamard=False, stream=None):
    """dsa_indexer_qk_prepare_store checked and bound once: returns a
    PreparedCall that launches it on these buffers (see PreparedCall)."""
    args, outs, _, _ = _qk_args(q, k, w, positions, out_cache_loc, cos_cache, sin_cache,
                                ln_gamma, ln_beta, ln_eps, softmax_scale, index_k_cache,
                                page_size, rope_dim, rope_style, q_fp8_out, weights_out,
                                num_tokens, max_position)
    fn = library().dsa_indexer_qk_prepare_store
    full = (*args, _flags(pdl, kernel) | _layout(cache_layout) | (FLAG_HADAMARD if hadamard else 0),
            _err_ptr(err_flags, q.device), _stream(stream, q.device))
    keep = (q, k, w, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta,
            index_k_cache, err_flags) + tuple(outs)
    return PreparedCall(fn, "dsa_indexer_qk_prepare_store", full, q.device, outs, keep)


def prepare_k_prepare_store(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta,
                            ln_eps, index_k_cache, page_size, rope_dim=64, rope_style=NEOX, *,
                            err_flags=None, num_tokens=None, max_position=None, pdl=False,
                            kernel="auto", cache_layout="paged", hadamard=False, stream=None):
    """dsa_indexer_k_prepare_store checked and bound once (see PreparedCall)."""
    args = _k_args(k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta, ln_eps,
                   index_k_cache, page_size, rope_dim, rope_style, num_tokens, max_position)
    fn = library().dsa_indexer_k_prepare_store
    full = (*args, _flags(pdl, kernel) | _layout(cache_layout) | (FLAG_HADAMARD if hadamard else 0),
            _err_ptr(err_flags, k.device), _stream(stream, k.device))
    keep = (k, positions, out_cache_loc, cos_cache, sin_cache, ln_gamma, ln_beta, index_k_cache,
            err_flags)
    return PreparedCall(fn, "dsa_indexer_k_prepare_store", full, k.device, None, keep)


def dsa_indexer_mqa_logits(q_fp8, weights, index_k_cache, page_size, block_table, context_lens,
                           max_context, *, logits=None, err_flags=None, pdl=False, stream=None):
    """fp8 paged MQA logits on the tensor cores:
    logits[t, j] = k_scale[j] * sum_h weights[t, h] * relu(q[t, h] . k[j])
    for j < context_lens[t], -inf up to max_context.  q_fp8 [T, H, 128]
    (float8_e4m3fn or uint8), weights [T, H] fp32, index_k_cache page-blocked
    (page_size 64), block_table [T, n >= ceil(max_context / 64)] int32 (the
    binding asks the table to cover max_context, so that no read of it can
    leave the tensor whatever the device-side context lengths are; contexts
    longer than max_context are clamped to it), context_lens [T] int32.
    ``pdl``: False, True, or "early" (PDL plus FLAG_PDL_EARLY_INDEX: the
    block table and context lengths are not written by the previous kernel).
    Returns logits [T, max_context] fp32."""
    if pdl not in (False, True, "early"):
        raise ValueError('pdl must be False, True or "early"')
    if q_fp8.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError("q_fp8 must be float8_e4m3fn or uint8 codes")
    if not q_fp8.is_cuda or not q_fp8.is_contiguous() or q_fp8.dim() != 3 \
            or q_fp8.shape[2] != HEAD_DIM:
        raise ValueError("q_fp8 must be a contiguous CUDA [T, H, 128] tensor")
    T, H = q_fp8.shape[0], q_fp8.shape[1]
    dev = q_fp8.device
    _need(weights, "weights", torch.float32, 2, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    if not isinstance(index_k_cache, torch.Tensor) or index_k_cache.device != dev:
        raise ValueError(f"index_k_cache must be a tensor on {dev}")
    if not weights.is_contiguous() or tuple(weights.shape) != (T, H):
        raise ValueError("weights must be contiguous [T, H]")
    if block_table.shape[0] < T or block_table.shape[1] * page_size < int(max_context):
        # every table read stays inside the tensor: contexts are clamped to max_context
        raise ValueError("block_table must be [T, >= ceil(max_context / page_size)]")
    if context_lens.shape[0] < T:
        raise ValueError(f"context_lens has fewer than {T} entries")
    if logits is None:
        logits = torch.empty((T, max(int(max_context), 1)), dtype=torch.float32, device=dev)
    _need(logits, "logits", torch.float32, 2, dev)
    if logits.shape[0] < T:
        raise ValueError(f"logits has fewer than {T} rows")
    with _on(q_fp8.device):
        st = library().dsa_indexer_mqa_logits(
            _ptr(q_fp8), _ptr(weights), _ptr(index_k_cache), _num_pages(index_k_cache, page_size),
            page_size, _ptr(block_table), block_table.stride(0), _ptr(context_lens), _ptr(logits),
            logits.stride(0), int(max_context), T, H,
            (FLAG_PDL if pdl else 0) | (FLAG_PDL_EARLY_INDEX if pdl == "early" else 0), _err_ptr(err_flags, q_fp8.device),
            _stream(stream, q_fp8.device))
    if st != 0:
        raise DsaError(st, "dsa_indexer_mqa_logits")
    return logits[:, :max_context]
