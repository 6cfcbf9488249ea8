"""An independent float64 restatement of the whole path for tiny inputs.

Used only by tests to pin the oracle (and never by the oracle): numpy
float64 LayerNorm, RoPE as complex multiplication, the scale exponent by
search over the integers, and the E4M3 code by nearest-value search over
CPU torch's float8_e4m3fn decode table with ties to the even code.  It rounds
nothing to fp32 on the way, so near a rounding boundary it may pick the other
neighbour; callers compare with that in mind.
"""
import numpy as np
import torch

_TABLE = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def code_of(v):
    m = abs(v)
    if m >= 448.0:
        c = 0x7E
    else:
        d = np.abs(_TABLE - m)
        best = np.flatnonzero(d == d.min())
        if best.size > 1:
            best = best[(best & 1) == 0]
        c = int(best[0])
    return c | (0x80 if (v < 0 and c != 0) else 0)


def exponent_of(amax):
    a = max(amax, float(np.float32(1e-4)))
    e = -200
    while a > 448.0 * 2.0 ** e:
        e += 1
    return e


def rope64(x, c, s, rope_dim, style):
    y = x.copy()
    half = rope_dim // 2
    i = np.arange(half)
    a, b = (i, i + half) if style == 0 else (2 * i, 2 * i + 1)
    z = (x[a] + 1j * x[b]) * (c[:half].astype(np.float64) + 1j * s[:half].astype(np.float64))
    y[a], y[b] = z.real, z.imag
    return y


def quant64(z):
    e = exponent_of(float(np.max(np.abs(z))))
    codes = np.array([code_of(v * 2.0 ** -e) for v in z], np.uint8)
    return codes, e


def bf16_round(v):
    """float64 values -> nearest bf16 (ties to even), as float64."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                    # v = m * 2^e, |m| in [0.5, 1)
    q = np.round(m * 256.0)               # 8 significant bits; np.round is ties-to-even
    return np.ldexp(q / 256.0, e)


def pipeline(inp, H=None, chain=False):
    """Returns (q_codes[T,H,128], q_exp[T,H], weights[T,H], k_codes[T,128],
    k_exp[T]) in float64 arithmetic.  chain=True rounds the LayerNorm output
    and the rotated vectors to bf16, as the four-launch chain does."""
    T = inp.T
    H = inp.H if H is None else H
    kb = inp.k_buffer().reshape(-1)
    wb = inp.kw.reshape(-1) if inp.kw is not None else inp.w.reshape(-1)
    w_off = 128 if inp.kw is not None else 0
    qc = np.zeros((T, H, 128), np.uint8)
    qe = np.zeros((T, H), np.int64)
    wt = np.zeros((T, H), np.float64)
    kc = np.zeros((T, 128), np.uint8)
    ke = np.zeros(T, np.int64)
    for t in range(T):
        p = inp.positions[t]
        c, s = inp.cos[p], inp.sin[p]
        for h in range(H):
            x = bf16(inp.q[t, h])
            z = rope64(x, c, s, inp.rope_dim, inp.style)
            if chain:
                z = bf16_round(z)
            qc[t, h], qe[t, h] = quant64(z)
            wv = bf16(wb[t * inp.w_stride_t + w_off + h])
            wt[t, h] = wv * 2.0 ** qe[t, h] * float(np.float32(inp.softmax_scale)) / np.sqrt(H)
        x = bf16(kb[t * inp.k_stride_t: t * inp.k_stride_t + 128])
        mu = x.mean()
        var = ((x - mu) ** 2).mean()
        y = (x - mu) / np.sqrt(var + float(np.float32(inp.eps))) * inp.gamma + inp.beta
        if chain:
            y = bf16_round(y)
        z = rope64(y, c, s, inp.rope_dim, inp.style)
        if chain:
            z = bf16_round(z)
        kc[t], ke[t] = quant64(z)
    return qc, qe, wt, kc, ke
