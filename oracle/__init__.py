"""Oracle for the DSA indexer Q/K prepare-and-store -- TEST INFRASTRUCTURE.

A plain, slow CPU statement of the path, written in C (``dsa_oracle.c``) and
loaded here through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package; the product
library never calls it and shares no code with it.

Every function cites the passage it restates in ``dsa_oracle.c``:
sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant + K-cache
write" (Motivation, Modifications, Accuracy) and vllm PR "[ROCm][Perf] Enable
fused indexer-Q RoPE+quant kernel for DeepSeek/GLM sparse attention" (Summary,
Kernel-level evidence), plus the OCP OFP8 spec for the E4M3 format.

Parity unpinned (stated readings, no pin from the pages): the 1e-4 amax
floor of the scale, the constants folded into the gate weights
(softmax_scale * H^-0.5) and the order LayerNorm-then-RoPE on k.  The
Hadamard rotation (``hadamard``) is pinned to the Sylvester matrix of scipy
and to a float64 brute force of the rotated pipeline.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_dsa.so")

NEOX, GPTJ = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no contraction of a*b+c into an fma)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.oracle_e4m3_encode.argtypes = [F32]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = F32
        lib.oracle_ue8m0_exponent.argtypes = [F32]
        lib.oracle_ue8m0_exponent.restype = ctypes.c_int
        lib.oracle_layernorm.argtypes = [P, P, P, F32, P]
        lib.oracle_layernorm.restype = None
        lib.oracle_rope.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int]
        lib.oracle_rope.restype = None
        lib.oracle_quantize_vector.argtypes = [P, P]
        lib.oracle_quantize_vector.restype = ctypes.c_int
        lib.oracle_k_prepare_store.argtypes = [
            I64, P, I64, P, P, P, P, I64, I64, P, P, F32, P, I64, I32, I32, I32, I32, P, I32]
        lib.oracle_k_prepare_store.restype = ctypes.c_int
        lib.oracle_qk_prepare_store.argtypes = [
            I64, I32, P, I64, I64, P, I64, P, I64, P, P, P, P, I64, I64, P, P, F32, F32,
            P, P, P, I64, I32, I32, I32, P, P, I32]
        lib.oracle_qk_prepare_store.restype = ctypes.c_int
        lib.oracle_qk_prepare_store_chain.argtypes = lib.oracle_qk_prepare_store.argtypes
        lib.oracle_qk_prepare_store_chain.restype = ctypes.c_int
        lib.oracle_qk_prepare_store_hadamard.argtypes = lib.oracle_qk_prepare_store.argtypes
        lib.oracle_qk_prepare_store_hadamard.restype = ctypes.c_int
        lib.oracle_hadamard.argtypes = [P]
        lib.oracle_hadamard.restype = None
        lib.oracle_mqa_logits.argtypes = [I32, I32, P, P, P, I64, I32, P, I64, P, P, I64, I32]
        lib.oracle_mqa_logits.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _req(a, dtype, writeable=False):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError("oracle arrays must be C-contiguous (pass strides separately)")
    if writeable and not a.flags.writeable:
        raise ValueError("output array is read-only")
    return a


# ------------------------------------------------------------- primitives

def e4m3_encode(v) -> np.ndarray:
    """fp32 values -> E4M3 codes (RNE, saturating), element by element."""
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, np.uint8)
    for i, x in enumerate(flat.tolist()):
        out[i] = lib.oracle_e4m3_encode(x)
    return out.reshape(v.shape)


def e4m3_decode(c) -> np.ndarray:
    """E4M3 codes -> fp32 values."""
    lib = _load()
    c = np.asarray(c, dtype=np.uint8)
    flat = c.reshape(-1)
    out = np.empty(flat.shape, np.float32)
    for i, x in enumerate(flat.tolist()):
        out[i] = lib.oracle_e4m3_decode(x)
    return out.reshape(c.shape)


def ue8m0_exponent(amax) -> np.ndarray:
    """Smallest e with max(amax, 1e-4) <= 448 * 2^e, element by element."""
    lib = _load()
    a = np.asarray(amax, dtype=np.float32)
    flat = a.reshape(-1)
    out = np.empty(flat.shape, np.int32)
    for i, x in enumerate(flat.tolist()):
        out[i] = lib.oracle_ue8m0_exponent(x)
    return out.reshape(a.shape)


def hadamard(x) -> np.ndarray:
    """Rows of x ([n, 128] fp32) -> H_128 x / sqrt(128), fp32 butterflies."""
    lib = _load()
    y = np.array(x, dtype=np.float32, copy=True, order="C").reshape(-1, 128)
    for i in range(y.shape[0]):
        lib.oracle_hadamard(_ptr(y[i]))
    return y


def layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """Row-wise LayerNorm of [n, 128] fp32 rows."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, 128)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    y = np.empty_like(x)
    for i in range(x.shape[0]):
        lib.oracle_layernorm(_ptr(x[i]), _ptr(gamma), _ptr(beta), eps, _ptr(y[i]))
    return y


def rope(x, cos_rows, sin_rows, rope_dim: int, style: int) -> np.ndarray:
    """Rotate the rope slice of each row of x ([n, D] fp32) by its own
    cos/sin row ([n, rope_dim/2] fp32)."""
    lib = _load()
    y = np.array(x, dtype=np.float32, copy=True, order="C")
    cos_rows = np.ascontiguousarray(cos_rows, dtype=np.float32)
    sin_rows = np.ascontiguousarray(sin_rows, dtype=np.float32)
    for i in range(y.shape[0]):
        lib.oracle_rope(_ptr(y[i]), _ptr(cos_rows[i]), _ptr(sin_rows[i]), rope_dim, style)
    return y


def quantize_vector(z) -> tuple[np.ndarray, int]:
    """One 128-vector -> (E4M3 codes, scale exponent e); scale = 2^e."""
    lib = _load()
    z = np.ascontiguousarray(z, dtype=np.float32).reshape(128)
    codes = np.empty(128, np.uint8)
    e = lib.oracle_quantize_vector(_ptr(z), _ptr(codes))
    return codes, e


# ------------------------------------------------------------- the path

def k_prepare_store(k, k_stride_t, positions, slots, cos_t, sin_t, cs_stride,
                    max_position, gamma, beta, eps, cache, num_pages, page_size,
                    rope_dim, style, bf16_intermediate=False, T=None, token_major=False):
    """k-only prepare-and-store.  ``k`` holds bf16 bit patterns (uint16) with
    row stride ``k_stride_t`` elements; ``cache`` (uint8) is written in place,
    page-blocked or (token_major) 132 bytes per slot.
    Returns (err_bits, k_scale_exp[T])."""
    lib = _load()
    positions = _req(positions, np.int64)
    slots = _req(slots, np.int64)
    T = len(positions) if T is None else T
    k = _req(k, np.uint16)
    cos_t, sin_t = _req(cos_t, np.float32), _req(sin_t, np.float32)
    gamma, beta = _req(gamma, np.float32), _req(beta, np.float32)
    cache = _req(cache, np.uint8, writeable=True)
    exps = np.zeros(max(T, 1), np.int32)
    err = lib.oracle_k_prepare_store(
        T, _ptr(k), k_stride_t, _ptr(positions), _ptr(slots), _ptr(cos_t), _ptr(sin_t),
        cs_stride, max_position, _ptr(gamma), _ptr(beta), eps, _ptr(cache), num_pages,
        page_size, rope_dim, style, int(bf16_intermediate), _ptr(exps), int(bool(token_major)))
    return err, exps[:T]


def qk_prepare_store(q, q_stride_t, q_stride_h, k, k_stride_t, w, w_stride_t,
                     positions, slots, cos_t, sin_t, cs_stride, max_position,
                     gamma, beta, eps, softmax_scale, q_fp8, weights, cache,
                     num_pages, page_size, H, rope_dim, style, T=None, chain=False,
                     token_major=False, hadamard=False):
    """Fused Q/K prepare-and-store.  q/k/w are bf16 bit patterns (uint16)
    with the given strides in elements.  ``q_fp8`` ([T, H, 128] uint8),
    ``weights`` ([T, H] fp32) and ``cache`` (uint8) are written in place.
    ``chain=True`` gives the outputs of the four-launch unfused chain, which
    rounds the LayerNorm output and the rotated vectors to bf16;
    ``hadamard=True`` rotates q heads and k by H_128 / sqrt(128) after RoPE.
    Returns (err_bits, q_scale_exp[T, H], k_scale_exp[T])."""
    lib = _load()
    positions = _req(positions, np.int64)
    slots = _req(slots, np.int64)
    T = len(positions) if T is None else T
    q, k, w = _req(q, np.uint16), _req(k, np.uint16), _req(w, np.uint16)
    cos_t, sin_t = _req(cos_t, np.float32), _req(sin_t, np.float32)
    gamma, beta = _req(gamma, np.float32), _req(beta, np.float32)
    q_fp8 = _req(q_fp8, np.uint8, writeable=True)
    weights = _req(weights, np.float32, writeable=True)
    cache = _req(cache, np.uint8, writeable=True)
    if q_fp8.size < T * H * 128 or weights.size < T * H:
        raise ValueError("output buffers too small")
    qe = np.zeros((max(T, 1), H), np.int32)
    ke = np.zeros(max(T, 1), np.int32)
    if chain and hadamard:
        raise ValueError("the chain has no Hadamard variant")
    fn = lib.oracle_qk_prepare_store_chain if chain else (
        lib.oracle_qk_prepare_store_hadamard if hadamard else lib.oracle_qk_prepare_store)
    err = fn(
        T, H, _ptr(q), q_stride_t, q_stride_h, _ptr(k), k_stride_t, _ptr(w), w_stride_t,
        _ptr(positions), _ptr(slots), _ptr(cos_t), _ptr(sin_t), cs_stride, max_position,
        _ptr(gamma), _ptr(beta), eps, softmax_scale, _ptr(q_fp8), _ptr(weights),
        _ptr(cache), num_pages, page_size, rope_dim, style, _ptr(qe), _ptr(ke),
        int(bool(token_major)))
    return err, qe[:T], ke[:T]


def mqa_logits(q_fp8, weights, cache, num_pages, page_size, block_table, context_lens,
               max_context):
    """fp8 paged MQA logits (the indexer's score for each (token, key)):
    logits[t, j] = k_scale[j] * sum_h weights[t, h] * max(q[t, h] . k[j], 0)
    for j < context_lens[t], -inf after.  q_fp8 [T, H, 128] uint8 codes,
    weights [T, H] fp32, cache page-blocked uint8, block_table [T, n] int32.
    Returns (err_bits, logits [T, max_context] fp32)."""
    lib = _load()
    q_fp8 = _req(q_fp8, np.uint8)
    T, H = q_fp8.shape[0], q_fp8.shape[1]
    weights = _req(weights, np.float32)
    cache = _req(cache, np.uint8)
    block_table = _req(block_table, np.int32)
    context_lens = _req(context_lens, np.int32)
    out = np.empty((max(T, 1), max(max_context, 1)), np.float32)
    err = lib.oracle_mqa_logits(T, H, _ptr(q_fp8), _ptr(weights), _ptr(cache), num_pages,
                                page_size, _ptr(block_table), block_table.shape[1],
                                _ptr(context_lens), _ptr(out), out.shape[1], max_context)
    return err, out[:T, :max_context]
