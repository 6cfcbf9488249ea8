"""Seeded synthetic inputs for the DSA indexer Q/K prepare-and-store.

The one module shared by the oracle side and the GPU side: it draws random
numbers and lays out buffers, and holds none of the method's arithmetic (no
LayerNorm, RoPE, scale or quantisation).  The RoPE cos/sin cache is an input of
the path (the serving engine's rope module owns it: sglang PR "[AMD] [GLM5]
Fuse the DSA indexer Q/K rope + quant + K-cache write", Modifications), so it
is built here: theta = pos * base^(-2i/rope_dim) in float64, cos/sin rounded
to fp32, one row of rope_dim/2 per position.

Workloads (shapes of the pages' serving benches: decode tokens per call =
concurrency 1..64, prefill T = input length 8192):
  tiny     T=4,  H=8,  NeoX, q/k/w ~N(0,1), positions U[0,4096), 4 pages of 64
  decode   T=64, H=64, GPT-J, k ~N(0,1)+0.5, positions U[0,131072), 4096 pages
  sweep    T in {1,8,32,64,256}, H=32, NeoX, k ~N(0,1)+0.5, positions
           U[0,262144), 4096 pages
  prefill  T=8192, H=64, NeoX, positions 0..8191, slots contiguous in 128 pages
  stress   T=65536 = 8 sequences x 8192, H=64, either pairing, q/k Student-t
           (nu=3) x 4, zero rows, planted e4m3 midpoints, shuffled page table
           of 2048 pages
All bf16 tensors are produced by round-to-nearest-even from fp32 draws.
"""
from __future__ import annotations

import dataclasses
import functools
from concurrent.futures import ThreadPoolExecutor

import numpy as np

D = 128
NEOX, GPTJ = 0, 1
ROPE_BASE = 10000.0
_CHUNK = 1 << 22


@dataclasses.dataclass
class Inputs:
    """Host buffers of one call.  q/k/w hold bf16 bit patterns (uint16).

    ``q`` is [T, H, 128] contiguous; ``k`` and ``w`` are views of ``kw``, a
    [T, 128 + H (padded to 8)] buffer laid out like the fused k/weights
    projection output (k in columns [0, 128), w in [128, 128 + H)), or separate
    contiguous buffers when ``kw`` is None.  Strides are in elements."""
    name: str
    T: int
    H: int
    rope_dim: int
    style: int
    page_size: int
    num_pages: int
    max_position: int
    q: np.ndarray
    k: np.ndarray
    w: np.ndarray
    positions: np.ndarray
    slots: np.ndarray
    cos: np.ndarray
    sin: np.ndarray
    gamma: np.ndarray
    beta: np.ndarray
    eps: float = 1e-6
    softmax_scale: float = float(np.float32(D ** -0.5))
    kw: np.ndarray | None = None
    token_major: bool = False   # index-K cache layout: 132 bytes per slot

    @property
    def q_stride_t(self):
        return self.H * D

    @property
    def q_stride_h(self):
        return D

    @property
    def k_stride_t(self):
        return self.kw.shape[1] if self.kw is not None else D

    @property
    def w_stride_t(self):
        return self.kw.shape[1] if self.kw is not None else self.H

    @property
    def cs_stride(self):
        return self.cos.shape[1]

    @property
    def cache_bytes(self):
        return self.num_pages * self.page_size * (D + 4)

    def k_buffer(self):
        """The buffer k's row stride refers to (flat start at k[0, 0])."""
        return self.kw if self.kw is not None else self.k



def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@functools.lru_cache(maxsize=8)
def rope_table(max_position: int, rope_dim: int, base: float = ROPE_BASE):
    """cos/sin cache [max_position, rope_dim/2] fp32 (angles in float64).
    Cached per arguments: callers must not modify the arrays."""
    half = rope_dim // 2
    inv_freq = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / rope_dim)
    theta = np.arange(max_position, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


def _chunked(seed_seq: np.random.SeedSequence, n: int, draw) -> np.ndarray:
    """Fill n float32 values chunk by chunk, each chunk from its own child
    seed, in a thread pool (numpy releases the GIL in its fills)."""
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    kids = seed_seq.spawn(nchunks)
    out = np.empty(n, np.float32)

    def work(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        out[lo:hi] = draw(np.random.Generator(np.random.PCG64(kids[i])), hi - lo)

    with ThreadPoolExecutor(8) as ex:
        list(ex.map(work, range(nchunks)))
    return out


def _normal(ss, n, offset=0.0):
    def draw(r, m):
        z = r.standard_normal(m, dtype=np.float32)
        return z + np.float32(offset) if offset else z
    return _chunked(ss, n, draw)


def _student_t(ss, n, nu=3.0, scale=4.0):
    def draw(r, m):
        z = r.standard_normal(m, dtype=np.float32)
        g = r.standard_gamma(nu / 2.0, m, dtype=np.float32)  # chi2_nu / 2
        return np.float32(scale) * z / np.sqrt(g * np.float32(2.0 / nu))
    return _chunked(ss, n, draw)


def _norm_params(rng):
    gamma = rng.uniform(0.5, 1.5, D).astype(np.float32)
    beta = (rng.standard_normal(D) * 0.1).astype(np.float32)
    return gamma, beta


def _distinct_slots(rng, T, num_pages, page_size):
    return rng.choice(num_pages * page_size, size=T, replace=False).astype(np.int64)


def _assemble(name, rng, ss, T, H, rope_dim, style, page_size, num_pages,
              max_position, q32, k32, positions, slots, fused_kw=True):
    w32 = _normal(ss.spawn(1)[0], T * H).reshape(T, H)
    gamma, beta = _norm_params(rng)
    cos, sin = rope_table(max_position, rope_dim)
    q = to_bf16_bits(q32).reshape(T, H, D)
    kb = to_bf16_bits(k32).reshape(T, D)
    wb = to_bf16_bits(w32).reshape(T, H)
    kw = None
    if fused_kw:
        # row length padded to 8 elements (16 bytes), as a GEMM output's
        # leading dimension is; the pad columns hold zeros
        kw = np.zeros((T, (D + H + 7) // 8 * 8), np.uint16)
        kw[:, :D] = kb
        kw[:, D:D + H] = wb
        kb, wb = kw[:, :D], kw[:, D:D + H]
    return Inputs(name=name, T=T, H=H, rope_dim=rope_dim, style=style,
                  page_size=page_size, num_pages=num_pages, max_position=max_position,
                  q=q, k=kb, w=wb, positions=positions.astype(np.int64),
                  slots=slots.astype(np.int64), cos=cos, sin=sin, gamma=gamma,
                  beta=beta, kw=kw)


def make_tiny(seed=0, T=4, H=8, style=NEOX, fused_kw=False):
    rng = np.random.default_rng(seed)
    ss = np.random.SeedSequence(seed)
    q32 = _normal(ss.spawn(1)[0], T * H * D)
    k32 = _normal(ss.spawn(1)[0], T * D)
    pos = rng.integers(0, 4096, T)
    slots = _distinct_slots(rng, T, 4, 64)
    return _assemble("tiny", rng, ss, T, H, 64, style, 64, 4, 4096, q32, k32, pos,
                     slots, fused_kw)


def make_decode(seed=1, T=64, H=64, style=GPTJ, max_position=131072, num_pages=4096,
                name="decode"):
    rng = np.random.default_rng(seed)
    ss = np.random.SeedSequence(seed)
    q32 = _normal(ss.spawn(1)[0], T * H * D)
    k32 = _normal(ss.spawn(1)[0], T * D, offset=0.5)
    pos = rng.integers(0, max_position, T)
    slots = _distinct_slots(rng, T, num_pages, 64)
    return _assemble(name, rng, ss, T, H, 64, style, 64, num_pages, max_position, q32,
                     k32, pos, slots)


def make_sweep(T, seed=2, H=32):
    return make_decode(seed=seed + 1000 * T, T=T, H=H, style=NEOX, max_position=262144,
                       name=f"sweep_T{T}")


def make_prefill(seed=3, T=8192, H=64, style=NEOX):
    rng = np.random.default_rng(seed)
    ss = np.random.SeedSequence(seed)
    q32 = _normal(ss.spawn(1)[0], T * H * D)
    k32 = _normal(ss.spawn(1)[0], T * D)
    pos = np.arange(T)
    num_pages = (T + 63) // 64
    slots = np.arange(T)
    return _assemble("prefill", rng, ss, T, H, 64, style, 64, num_pages, T, q32, k32,
                     pos, slots)


def e4m3_midpoints() -> np.ndarray:
    """The 126 positive values halfway between adjacent finite E4M3 codes,
    from the OFP8 E4M3 definition (bias 7, subnormal step 2^-9, max 448)."""
    vals = [m * 2.0 ** -9 for m in range(8)]
    vals += [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)
             if not (e == 15 and m == 7)]
    vals = np.array(vals)
    return ((vals[:-1] + vals[1:]) / 2).astype(np.float32)


def make_stress(seed=4, style=NEOX, n_seq=8, seq_len=8192, H=64, pages=2048):
    """Heavy-tailed prefill with planted edge cases.

    * q and k ~ Student-t(nu=3) x 4, rounded to bf16;
    * one q head row in 1024 and one k row in 1024 all zero (at least one each);
    * in a quarter of the q head rows ("planted rows"): the row is rescaled so
      one pass-through element (dim >= rope_dim, untouched by RoPE) is exactly
      +-448 * 2^e and every other element has magnitude <= 224 * 2^e, which
      makes 2^e the row's scale whatever the rotation does; then about five
      other pass-through elements are set to +-m * 2^e with m an E4M3 midpoint
      below 448, so they reach the quantiser as exact ties (about 1% of all q
      elements);
    * 1% of k elements are set to +-m * 2^j (m a midpoint, j in [-3, 0]) at the
      input; LayerNorm and RoPE move them off the tie, so they only make
      near-ties;
    * slots: sequence s, token j -> page_table[s][j // 64] * 64 + j % 64 over a
      shuffled permutation of the page pool.
    """
    T = n_seq * seq_len
    rng = np.random.default_rng(seed)
    ss = np.random.SeedSequence(seed)
    q32 = _student_t(ss.spawn(1)[0], T * H * D).reshape(T * H, D)
    k32 = _student_t(ss.spawn(1)[0], T * D).reshape(T, D)
    rope_dim = 64
    mids = e4m3_midpoints()

    # planted rows of q
    rows = np.flatnonzero(rng.random(T * H) < 0.25)
    sub = q32[rows]
    # round the row to bf16 first so the bound below holds on the stored values
    sub = bf16_bits_to_f32(to_bf16_bits(sub))
    m = np.abs(sub).max(axis=1)
    m = np.maximum(m, np.float32(1e-3))
    e = np.ceil(np.log2(2.0 * m.astype(np.float64) / 448.0)).astype(np.int64)
    anchor = rng.integers(rope_dim, D, rows.size)
    sign = np.where(rng.random(rows.size) < 0.5, -1.0, 1.0)
    sub[np.arange(rows.size), anchor] = (sign * 448.0 * np.exp2(e)).astype(np.float32)
    n_mid = 5
    for _ in range(n_mid):
        col = rng.integers(rope_dim, D, rows.size)
        ok = col != anchor
        mv = mids[rng.integers(0, mids.size - 1, rows.size)].astype(np.float64)  # < 448
        sg = np.where(rng.random(rows.size) < 0.5, -1.0, 1.0)
        val = (sg * mv * np.exp2(e)).astype(np.float32)
        r_ok = np.flatnonzero(ok)
        sub[r_ok, col[r_ok]] = val[r_ok]
    q32[rows] = sub

    # near-ties on k
    kmask = rng.random(k32.shape) < 0.01
    nk = int(kmask.sum())
    k32[kmask] = (np.where(rng.random(nk) < 0.5, -1.0, 1.0)
                  * mids[rng.integers(0, 120, nk)].astype(np.float64)
                  * np.exp2(rng.integers(-3, 1, nk))).astype(np.float32)

    # zero rows (never a planted row, so the plant stays intact)
    planted = np.zeros(T * H, bool)
    planted[rows] = True
    zq = np.flatnonzero((rng.random(T * H) < 1.0 / 1024) & ~planted)
    if zq.size == 0:
        zq = np.flatnonzero(~planted)[:1]
    q32[zq] = 0.0
    zk = np.flatnonzero(rng.random(T) < 1.0 / 1024)
    if zk.size == 0:
        zk = np.array([0])
    k32[zk] = 0.0

    positions = np.tile(np.arange(seq_len), n_seq)
    perm = rng.permutation(pages)
    pages_per_seq = seq_len // 64
    seq = np.repeat(np.arange(n_seq), seq_len)
    j = positions
    slots = perm[seq * pages_per_seq + j // 64] * 64 + j % 64
    inp = _assemble("stress", rng, ss, T, H, rope_dim, style, 64, pages, seq_len,
                    q32.reshape(-1), k32.reshape(-1), positions, slots)
    inp.planted_rows = rows
    inp.planted_exp = e
    inp.zero_q_rows = zq
    inp.zero_k_rows = zk
    return inp


def make_k_bulk(seed=6, style=NEOX, n_seq=8, seq_len=8192, H=64, pages=2048):
    """The k-only call (the index-K store of the dense fast path) at prefill
    size: the stress set's keys without the query side.  Keys ~ Student-t(3)
    x 4 rounded to bf16, 1% of elements set to +-m * 2^j (m an E4M3 midpoint,
    j in [-3, 0]), 1/1024 rows all zero (at least one); positions 0..seq_len-1
    in each of n_seq sequences; slots through a shuffled page table.  k sits
    in the fused [T, 128 + H] k|w projection layout (w ~ N(0,1)); q is empty."""
    T = n_seq * seq_len
    rng = np.random.default_rng(seed)
    ss = np.random.SeedSequence(seed)
    k32 = _student_t(ss.spawn(1)[0], T * D).reshape(T, D)
    mids = e4m3_midpoints()
    kmask = rng.random(k32.shape) < 0.01
    nk = int(kmask.sum())
    k32[kmask] = (np.where(rng.random(nk) < 0.5, -1.0, 1.0)
                  * mids[rng.integers(0, 120, nk)].astype(np.float64)
                  * np.exp2(rng.integers(-3, 1, nk))).astype(np.float32)
    zk = np.flatnonzero(rng.random(T) < 1.0 / 1024)
    k32[zk if zk.size else np.array([0])] = 0.0
    w32 = _normal(ss.spawn(1)[0], T * H).reshape(T, H)
    kw = np.zeros((T, (D + H + 7) // 8 * 8), np.uint16)
    kw[:, :D] = to_bf16_bits(k32)
    kw[:, D:D + H] = to_bf16_bits(w32)
    positions = np.tile(np.arange(seq_len), n_seq).astype(np.int64)
    perm = rng.permutation(pages)
    seq = np.repeat(np.arange(n_seq), seq_len)
    slots = (perm[seq * (seq_len // 64) + positions // 64] * 64 + positions % 64).astype(np.int64)
    gamma, beta = _norm_params(rng)
    cos, sin = rope_table(seq_len, 64)
    return Inputs(name="k_bulk", T=T, H=H, rope_dim=64, style=style, page_size=64,
                  num_pages=pages, max_position=seq_len, q=np.zeros((0, H, D), np.uint16),
                  k=kw[:, :D], w=kw[:, D:D + H], positions=positions, slots=slots, cos=cos,
                  sin=sin, gamma=gamma, beta=beta, kw=kw)


CONFIGS = {
    "tiny": make_tiny,
    "decode": make_decode,
    "prefill": make_prefill,
    "stress": make_stress,
}


def algorithmic_bytes(T: int, H: int, with_q: bool = True) -> int:
    """Bytes one call must move: reads q, k, w, position, slot, the cos/sin
    row and gamma/beta; writes q_fp8, fp32 weights, 128 code bytes and one
    fp32 scale per token."""
    if with_q:
        return T * (3 * H * D + 6 * H + 660) + 1024
    return T * 660 + 1024


@dataclasses.dataclass
class LogitsInputs:
    """Inputs of the indexer's fp8 paged MQA logits (the consumer of this
    path's outputs): q codes [T, H, 128] (uint8 e4m3), gate weights [T, H]
    fp32, a page-blocked index-K cache, per-token block tables and context
    lengths."""
    T: int
    H: int
    page_size: int
    num_pages: int
    q_fp8: np.ndarray
    weights: np.ndarray
    cache: np.ndarray
    block_table: np.ndarray
    context_lens: np.ndarray
    max_context: int


def random_e4m3_codes(rng, shape, max_exp_field=11):
    """Uniform random finite e4m3 codes with exponent field <= max_exp_field
    (so |value| <= 2^(max_exp_field - 6)), either sign; no NaN codes."""
    mag = rng.integers(0, (max_exp_field + 1) * 8, size=shape, dtype=np.int64)
    sign = rng.integers(0, 2, size=shape, dtype=np.int64) << 7
    return (mag | sign).astype(np.uint8)


def make_logits(seed=5, T=64, H=64, context=16384, page_size=64, ragged=False, spare_pages=0):
    """Decode-step logits workload: T sequences (one query token each, H
    indexer heads) with `context` cached keys each (or, ragged, uniform in
    [1, context]), every sequence on its own shuffled pages; scales are
    powers of two 2^e, e uniform in [-10, 0]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, context + 1, T) if ragged else np.full(T, context)
    blocks = (lens + page_size - 1) // page_size
    num_pages = int(blocks.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_blocks = int(blocks.max())
    table = np.zeros((T, max_blocks), np.int32)
    at = 0
    for t in range(T):
        table[t, :blocks[t]] = perm[at:at + blocks[t]]
        at += blocks[t]
    cache = np.empty((num_pages, page_size * (D + 4)), np.uint8)
    cache[:, :page_size * D] = random_e4m3_codes(rng, (num_pages, page_size * D))
    exps = rng.integers(-10, 1, (num_pages, page_size)).astype(np.uint32)
    cache[:, page_size * D:] = ((exps + np.uint32(127)) << np.uint32(23)).view(np.uint8).reshape(
        num_pages, page_size * 4)
    q = random_e4m3_codes(rng, (T, H, D))
    w = (rng.standard_normal((T, H)) * 0.05).astype(np.float32)
    return LogitsInputs(T=T, H=H, page_size=page_size, num_pages=num_pages, q_fp8=q, weights=w,
                        cache=cache.reshape(-1), block_table=table,
                        context_lens=lens.astype(np.int32), max_context=int(lens.max()))
