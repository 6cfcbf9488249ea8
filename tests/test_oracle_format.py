"""Pins of the oracle's E4M3 encoder/decoder and ue8m0 scale rule.

Each pin comes from outside the oracle: the OFP8 specification's special
values (golden file), CPU torch's float8_e4m3fn (a library routine),
brute-force nearest-code search, and brute force over the exponent range.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

_POS_CODES = np.arange(127, dtype=np.uint8)  # finite non-negative codes


def _torch_decode(codes):
    t = torch.tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _nearest_code(v, table):
    """Nearest finite E4M3 code to v by search; ties to the even code;
    saturate beyond 448 (the sign is applied afterwards)."""
    m = abs(float(v))
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    if m >= 448.0:
        return sign | 0x7E
    d = np.abs(table - m)
    best = np.flatnonzero(d == d.min())
    if best.size > 1:
        best = best[(best & 1) == 0]
    return sign | int(best[0])


def test_ofp8_golden_points(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "ofp8_e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                v, c = line.split()
                rows.append((float(v), int(c, 16)))
    assert len(rows) >= 10
    for v, c in rows:
        assert oracle.e4m3_encode([v])[0] == c, (v, hex(c))
        assert oracle.e4m3_decode([c])[0] == np.float32(v), (v, hex(c))


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes).astype(np.float64)
    ref = _torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])


def test_encode_exhaustive_over_bf16():
    """Every finite bf16 value, alone and scaled into the E4M3 range."""
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    table = _torch_decode(_POS_CODES)
    # bring every value into [2^-12, 2^9) so all binades of E4M3 are hit
    with np.errstate(over="ignore"):
        e = np.floor(np.log2(np.maximum(np.abs(vals.astype(np.float64)), 1e-300)))
    shift = np.where(np.abs(vals) > 0, -12 - np.mod(e, 21), 0)
    scaled = (vals.astype(np.float64) * np.exp2(shift)).astype(np.float32)
    for arr in (vals, scaled):
        got = oracle.e4m3_encode(arr)
        exp = np.array([_nearest_code(v, table) for v in arr.tolist()], np.uint8)
        # the sign of zero is free for values that round to zero
        both_zero = ((got & 0x7F) == 0) & ((exp & 0x7F) == 0)
        assert np.array_equal(got[~both_zero], exp[~both_zero])


def test_encode_midpoints_tie_to_even():
    table = _torch_decode(_POS_CODES)
    mids = (table[:-1] + table[1:]) / 2
    assert mids.size == 126
    v = np.concatenate([mids, -mids]).astype(np.float32)
    assert np.array_equal(v.astype(np.float64), np.concatenate([mids, -mids]))
    got = oracle.e4m3_encode(v)
    lo = np.concatenate([np.arange(126), np.arange(126)])
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    even[126:] |= 0x80
    got_mag = got & 0x7F
    assert np.array_equal(got_mag, even & 0x7F)
    nz = got_mag != 0
    assert np.array_equal(got[nz] & 0x80, even[nz] & 0x80)


def test_encode_matches_torch_random():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(20000) * 50,
        rng.uniform(-464, 464, 20000),
        rng.standard_normal(20000) * 0.01,
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    both_zero = ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert np.array_equal(got[~both_zero], ref[~both_zero])


def test_encode_saturates_never_nan():
    v = np.array([448.0, 463.99, 464.0, 500.0, 1e30, -1e30, -470.0], np.float32)
    got = oracle.e4m3_encode(v)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def _brute_exponent(a):
    a = max(float(np.float32(a)), float(np.float32(1e-4)))
    for e in range(-140, 141):
        if a <= 448.0 * 2.0 ** e:
            return e
    raise AssertionError


def test_ue8m0_bruteforce():
    rng = np.random.default_rng(5)
    logu = np.exp(rng.uniform(np.log(1e-9), np.log(3e38), 4000)).astype(np.float32)
    bounds = []
    for k in range(-30, 127):
        b = np.float32(448.0 * 2.0 ** k) if 448.0 * 2.0 ** k < 3.4e38 else None
        if b is None or not np.isfinite(b):
            continue
        bounds += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    specials = np.array([0.0, 1e-4, np.nextafter(np.float32(1e-4), np.float32(0)),
                         np.nextafter(np.float32(1e-4), np.float32(1)), 1.0, 448.0],
                        np.float32)
    a = np.concatenate([logu, np.array(bounds, np.float32), specials])
    a = a[np.isfinite(a)]
    got = oracle.ue8m0_exponent(a)
    exp = np.array([_brute_exponent(x) for x in a.tolist()])
    assert np.array_equal(got, exp)
    # the scale is a power of two: fp32 bits have an empty mantissa
    scale = np.ldexp(np.float32(1), got).astype(np.float32)
    assert np.all((scale.view(np.uint32) & 0x7FFFFF) == 0)
    assert np.all(np.maximum(a.astype(np.float64), float(np.float32(1e-4))) <= 448.0 * np.exp2(got))


def test_ue8m0_floor_and_range():
    assert oracle.ue8m0_exponent([0.0])[0] == -22
    assert oracle.ue8m0_exponent([3.3895314e38])[0] == 120
    assert oracle.ue8m0_exponent([448.0])[0] == 0
    assert oracle.ue8m0_exponent([np.nextafter(np.float32(448), np.float32(1e3))])[0] == 1


def test_quantiser_is_scale_equivariant_and_odd():
    """Scaling a vector by 2^k leaves its codes alone and moves its exponent by
    k (while amax stays above the 1e-4 floor); negating it flips only the sign
    bits.  An exponent off by one, a scale applied twice or a sign dropped in
    the encoder breaks one of these."""
    rng = np.random.default_rng(41)
    for _ in range(200):
        z = (rng.standard_t(3, 128) * rng.uniform(0.01, 100)).astype(np.float32)
        codes, e = oracle.quantize_vector(z)
        for k in (-7, -1, 1, 5):
            zk = (z.astype(np.float64) * 2.0 ** k).astype(np.float32)
            if np.max(np.abs(zk)) <= 1e-4:
                continue
            ck, ek = oracle.quantize_vector(zk)
            assert ek == e + k and np.array_equal(ck, codes), k
        cn, en = oracle.quantize_vector(-z)
        assert en == e
        nonzero = codes & 0x7F != 0
        assert np.array_equal(cn[nonzero], codes[nonzero] ^ 0x80)
