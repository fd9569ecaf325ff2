"""Pins of the oracle's number-format codecs against library conversions and
brute-force nearest-value search (the formats' own definitions)."""
import numpy as np
import pytest
import torch

import oracle


def _table(decode_all):
    """(codes, values) of all finite non-negative codes, sorted by value."""
    codes = np.arange(decode_all[1], dtype=np.int64)
    vals = decode_all[0](codes)
    keep = np.isfinite(vals) & ~np.signbit(vals)
    order = np.argsort(vals[keep], kind="stable")
    return codes[keep][order], vals[keep][order]


def _torch_decode(dtype, n):
    def f(codes):
        if dtype == torch.float8_e4m3fn:
            t = torch.tensor(codes, dtype=torch.uint8).view(dtype)
        else:
            t = torch.tensor(codes.astype(np.uint16).view(np.int16)).view(dtype)
        return t.to(torch.float64).numpy()
    return f, n


def brute_nearest(x, codes, vals, overflow_to=None, overflow_at=None):
    """Nearest representable value to each double in x (ties to the even
    code); magnitudes at or past `overflow_at` give `overflow_to`."""
    out = []
    for v in np.asarray(x, np.float64):
        a = abs(v)
        if overflow_at is not None and a >= overflow_at:
            out.append(overflow_to if v > 0 else overflow_to | (0x8000 if overflow_to > 0xff else 0x80))
            continue
        i = np.searchsorted(vals, a)
        cands = [j for j in (i - 1, i) if 0 <= j < len(vals)]
        best = min(cands, key=lambda j: (abs(vals[j] - a), codes[j] & 1))
        c = int(codes[best])
        if np.signbit(v):
            c |= 0x8000 if len(codes) > 300 else 0x80
        out.append(c)
    return np.array(out)


def test_f16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_f64(codes)
    ref = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_to_f64(codes)
    ref = torch.tensor(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7e] == 448.0 and ours[0x01] == 2.0 ** -9


def _midpoints(vals):
    v = vals[np.isfinite(vals)]
    return (v[1:] + v[:-1]) / 2.0


def test_f16_encode_from_double():
    rng = np.random.default_rng(1)
    _, vals = _table(_torch_decode(torch.float16, 65536))
    mids = _midpoints(vals)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        mids[::7], -mids[::11], np.nextafter(mids[::13], np.inf), np.nextafter(mids[::13], -np.inf),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -25, 2.0 ** -24 * 1.5,
         1 + 2.0 ** -11 + 2.0 ** -40]])
    ours = oracle.f16_from_f64(x)
    ref = x.astype(np.float16).view(np.uint16)  # numpy rounds double -> half directly
    assert np.array_equal(ours, ref)


def test_bf16_encode_from_double_brute_force():
    rng = np.random.default_rng(2)
    codes, vals = _table(_torch_decode(torch.bfloat16, 65536))
    mids = _midpoints(vals)
    maxv = vals[-1]
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
        mids[::41], np.nextafter(mids[::53], np.inf), -np.nextafter(mids[::53], -np.inf),
        [1 + 2.0 ** -8 + 2.0 ** -40, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -133 * 1.5]])
    ours = oracle.bf16_from_f64(x)
    # values at or past max + half an ulp round to infinity
    ref = brute_nearest(x, codes, vals, overflow_to=0x7f80, overflow_at=maxv + 2.0 ** 119)
    assert np.array_equal(ours.astype(np.int64), ref)


def test_bf16_encode_matches_torch_on_float32():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    x = np.concatenate([x, np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8], np.float32)])
    ours = oracle.bf16_from_f64(x.astype(np.float64))
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_satfinite():
    rng = np.random.default_rng(4)
    codes, vals = _table(_torch_decode(torch.float8_e4m3fn, 256))
    mids = _midpoints(vals).astype(np.float32)
    x = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 3, 20000)).astype(np.float32),
        mids, -mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf)),
        np.array([448, 449, 463.9, 464, 464.1, 479, 480, 1e30, np.inf, -np.inf, -464, 2.0 ** -10,
                  3 * 2.0 ** -10, 0.0, -0.0], np.float32)])
    ours = oracle.e4m3_from_f32(x)
    clamped = np.clip(x.astype(np.float64), -448.0, 448.0)
    ref = brute_nearest(clamped, codes, vals)
    assert np.array_equal(ours.astype(np.int64), ref)
    # torch's non-saturating cast agrees once the input is clamped
    tref = torch.tensor(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, tref)
    assert oracle.e4m3_from_f32(np.array([np.nan], np.float32))[0] & 0x7f == 0x7f


def test_e4m3_roundtrip_identity_on_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    back = oracle.e4m3_from_f32(vals)
    # +0 and -0 both map to themselves
    assert np.array_equal(back, codes)
