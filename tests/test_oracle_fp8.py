"""Pins for the oracle's fp8 (e4m3) KV cache encoding and its attention.

The encoding is this library's own definition (the benchmarking blog on a
hosted 1M-context model, section 1, names a narrow-float KV cache as the
lever on decode bytes but gives no format): per cache row a binary32 scale
s = max|x| / 448 and codes e4m3(x / s), rounded to nearest even with
saturation.  The e4m3 conversion is pinned against PyTorch's float8_e4m3fn
(a library routine, on the values it does not saturate) and hand-derived
ties; the row encoder by a hand-worked row, exact round trips of rows that
are already on the grid, and the format's error bound; the fp8 attention by
its reduction to the bf16 definition when the encoding is exact.
"""
import numpy as np
import pytest
import torch

import workloads as W


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def torch_e4m3(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_values_match_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    # format facts: largest finite 448, smallest subnormal 2^-9, NaN only at 0x7F / 0xFF
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0**-9 and ours[0x08] == 2.0**-6
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and np.isnan(ours).sum() == 2


def test_float_to_e4m3_matches_torch(oracle):
    rng = np.random.default_rng(3)
    mags = np.exp2(rng.uniform(-13, 9, 20000)).astype(np.float32)
    x = mags * rng.choice([-1.0, 1.0], mags.size).astype(np.float32)
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    np.testing.assert_array_equal(oracle.float_to_e4m3(x), torch_e4m3(x))


def test_float_to_e4m3_ties_to_even_and_saturation(oracle):
    vals = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448, increasing
    assert np.all(np.diff(vals) > 0)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact in binary32
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)
    lower = np.arange(0x7E, dtype=np.uint8)
    want = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)  # even mantissa wins a tie
    np.testing.assert_array_equal(oracle.float_to_e4m3(mids), want)
    np.testing.assert_array_equal(oracle.float_to_e4m3(-mids), want | 0x80)
    np.testing.assert_array_equal(torch_e4m3(mids), want)
    # beyond the largest finite value the encoder saturates (no infinity in e4m3)
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e5, np.inf, -500.0, -np.inf], np.float32)
    np.testing.assert_array_equal(oracle.float_to_e4m3(big), [0x7E] * 6 + [0xFE] * 2)
    assert oracle.float_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    # signed zeros and the subnormal boundary: 2^-10 ties to 0, 3 * 2^-10 ties up to 2 * 2^-9
    np.testing.assert_array_equal(
        oracle.float_to_e4m3(np.array([0.0, -0.0, 2**-10, 3 * 2**-10, 2**-11, 2**-9 * 0.75], np.float32)),
        [0x00, 0x80, 0x00, 0x02, 0x00, 0x01])


def row_bits(vals, d):
    x = np.zeros(d, np.float32)
    x[: len(vals)] = vals
    return bits(torch.tensor(x).to(torch.bfloat16)).reshape(1, 1, 1, d)


def test_quantize_row_by_hand(oracle):
    # a = 2, s = fl(2 / 448); x / s rounds to 112, -224, 56, 448, 0 whose codes are
    # 112 = 1.75 * 2^6 -> (6 + 7) << 3 | 6 = 0x6E,  224 -> 0x76 | sign,  56 -> 0x66,  448 -> 0x7E
    codes, sc = oracle.quantize_kv_fp8(row_bits([0.5, -1.0, 0.25, 2.0], 8))
    assert sc.ravel()[0] == np.float32(2.0) / np.float32(448.0)
    assert list(codes.ravel()) == [0x6E, 0xF6, 0x66, 0x7E, 0, 0, 0, 0]
    # an all-zero row: scale 0 and zero codes (no division by zero)
    codes, sc = oracle.quantize_kv_fp8(row_bits([], 8))
    assert sc.ravel()[0] == 0.0 and not codes.any()
    # signed zeros keep their sign bit: -0 / s = -0 -> 0x80
    codes, _ = oracle.quantize_kv_fp8(row_bits([1.0, -0.0], 4))
    assert list(codes.ravel()) == [0x7E, 0x80, 0, 0]


def grid_cache(rng, B, H, L, d):
    """Rows whose values are e4m3 grid points times a power of two, with one
    entry of magnitude exactly 448 * 2^-k: their encoding is exact."""
    c = rng.integers(0, 0x7E, size=(B, H, L, d)).astype(np.uint8)
    c |= (rng.integers(0, 2, size=c.shape) << 7).astype(np.uint8)
    c[..., 0] = np.where(rng.integers(0, 2, size=(B, H, L)) == 1, 0x7E, 0xFE)
    k = rng.integers(-6, 9, size=(B, H, L)).astype(np.float64)
    vals = torch.tensor(c).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.exp2(-k)[..., None]
    x = bits(torch.tensor(vals).to(torch.bfloat16))
    assert np.array_equal((x.astype(np.uint32) << 16).view(np.float32).astype(np.float64), vals)
    return x, c, np.exp2(-k).astype(np.float32)


def test_exact_round_trip(oracle):
    rng = np.random.default_rng(5)
    x, c, s = grid_cache(rng, 2, 3, 40, 64)
    codes, sc = oracle.quantize_kv_fp8(x)
    np.testing.assert_array_equal(sc, s)
    np.testing.assert_array_equal(codes, c)
    deq = oracle.dequantize_kv_fp8(codes, sc)
    np.testing.assert_array_equal(deq, (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


def test_error_bound_and_row_max(oracle):
    rng = np.random.default_rng(6)
    B, H, L, d = 2, 2, 50, 128
    mag = np.exp2(rng.uniform(-30, 30, size=(B, H, L, 1)))
    xf = rng.standard_normal((B, H, L, d)) * mag
    x = bits(torch.tensor(xf, dtype=torch.float32).to(torch.bfloat16))
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, sc = oracle.quantize_kv_fp8(x)
    deq = oracle.dequantize_kv_fp8(codes, sc)
    s = sc.astype(np.float64)[..., None]
    # half a unit in the last place of e4m3 (2^-4 relative, 2^-10 absolute for
    # subnormals) of x / s, plus the binary32 roundings of s and x / s
    bound = (2.0**-4 * np.abs(xv) + 2.0**-10 * s) * (1 + 2.0**-20)
    assert np.all(np.abs(deq - xv) <= bound)
    # every row's largest entry lands on +-448 exactly
    vmax = np.abs(oracle.e4m3_value(codes.ravel()).reshape(codes.shape)).max(axis=-1)
    assert np.all(vmax == 448.0)
    assert np.all(np.signbit(deq) == np.signbit(xv))


def test_rows_past_seq_len_untouched(oracle):
    rng = np.random.default_rng(7)
    x = bits(torch.randn(2, 2, 30, 64).to(torch.bfloat16))
    sl = np.array([17, 0], np.int32)
    codes, sc = oracle.quantize_kv_fp8(x, sl)
    assert not codes[0, :, 17:].any() and not sc[0, :, 17:].any() and not codes[1].any()
    full, fsc = oracle.quantize_kv_fp8(x)
    np.testing.assert_array_equal(codes[0, :, :17], full[0, :, :17])
    np.testing.assert_array_equal(sc[0, :, :17], fsc[0, :, :17])
    with pytest.raises(ValueError):
        oracle.quantize_kv_fp8(x, np.array([31, 0], np.int32))


def test_fp8_attention_reduces_to_bf16_when_exact(oracle):
    rng = np.random.default_rng(8)
    B, Hq, Hkv, L, d = 2, 4, 2, 70, 64
    k, kc, ks = grid_cache(rng, B, Hkv, L, d)
    v, vc, vs = grid_cache(rng, B, Hkv, L, d)
    q = bits(torch.randn(B, Hq, d).to(torch.bfloat16))
    sl = np.array([70, 33], np.int32)
    out8, lse8 = oracle.decode_dense_fp8(q, kc, ks, vc, vs, sl, 0.02)
    out, lse = oracle.decode_dense(q, k, v, sl, 0.02)
    np.testing.assert_allclose(out8, out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse8, lse, rtol=1e-13, atol=1e-13)


def test_fp8_attention_error_follows_encoding(oracle):
    # on a realistic cache, the fp8 result sits within the output tolerance of
    # the bf16 result (the encoding moves each K/V entry by <= 2^-4 relative)
    p = W.random_problem(B=1, Hq=4, Hkv=2, d=128, L_max=300, seed=9)
    kc, ks = oracle.quantize_kv_fp8(p.k)
    vc, vs = oracle.quantize_kv_fp8(p.v)
    out8, _ = oracle.decode_dense_fp8(p.q, kc, ks, vc, vs, None, p.scale)
    out, _ = oracle.decode_dense(p.q, p.k, p.v, None, p.scale)
    err = np.abs(out8 - out)
    assert err.max() < 0.05 * (1 + np.abs(out).max())
    assert err.max() > 0  # the encoding is lossy here
