"""Pins for the oracle's fp4 (e2m1) KV cache encoding and its attention.

The encoding is this library's own definition (the benchmarking blog on a
hosted 1M-context model, section 1, names an "FP4" KV cache but gives no
format): per cache row and 32-channel block a power-of-two scale 2^e, e the
smallest integer in [-126, 127] with 6 * 2^e >= the block's max |x|, and
e2m1 codes of x * 2^-e (round to nearest, ties to even).  Pinned by the
format's value table, hand-worked ties and rows, an independent rounding
formula (numpy's round-half-even on the e2m1 quantum of each binade), the
exponent's closed form in exact rational arithmetic, exact round trips of
on-grid rows, the error bound, and the reduction of the fp4 attention to
the bf16 definition when the encoding is exact.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table(oracle):
    vals = oracle.e2m1_value(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(vals[:8], E2M1)
    np.testing.assert_array_equal(vals[8:], [-v for v in E2M1])
    assert math.copysign(1.0, vals[8]) == -1.0  # code 8 is -0


def test_ties_and_saturation_by_hand(oracle):
    # midpoints between neighbours go to the code with mantissa bit 0 (even code)
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.2499: 0, 0.2501: 1, 0.7: 1, 4.99: 6, 5.01: 7, 6.0: 7, 7.0: 7, 1e30: 7, 0.0: 0}
    got = oracle.to_e2m1(list(cases))
    assert list(got) == list(cases.values())
    neg = oracle.to_e2m1([-k for k in cases])
    assert list(neg) == [v | 8 for v in cases.values()]


def rne_grid(y):
    """Independent formula: RNE on the e2m1 quantum of y's binade (0.5 below 2,
    then 2^(floor(log2|y|) - 1)), numpy's round-half-even, saturating at 6."""
    a = np.abs(y)
    k = np.floor(np.log2(np.maximum(a, 1e-300)))
    q = np.exp2(np.maximum(k, 0.0) - 1.0)
    v = np.minimum(np.round(a / q) * q, 6.0)
    return np.where(np.signbit(y), -v, v)


def test_rounding_matches_independent_formula(oracle):
    rng = np.random.default_rng(11)
    y = np.concatenate([rng.uniform(-7, 7, 20000), np.arange(-6.5, 6.51, 0.125), rng.uniform(-0.3, 0.3, 2000)])
    codes = oracle.to_e2m1(y)
    np.testing.assert_array_equal(oracle.e2m1_value(codes), rne_grid(y))


def exact_exponent(amax):
    """Smallest integer e in [-126, 127] with 6 * 2^e >= amax, by exact rationals."""
    a = Fraction(amax)
    e = -126
    while e < 127 and Fraction(6) * Fraction(2) ** e < a:
        e += 1
    return e


def test_block_exponent_closed_form(oracle):
    rng = np.random.default_rng(12)
    amaxes = [0.0, 6.0, 3.0, 1.5, 12.0, 6.0 * 2.0**-126, 6.0 * 2.0**-127, 1e-40, 3.0e38]
    for k in range(-20, 21):
        b = 6.0 * 2.0**k
        amaxes += [b, np.nextafter(b, 0.0), np.nextafter(b, np.inf)]
    amaxes += list(np.exp2(rng.uniform(-60, 60, 500)))
    for a in amaxes:
        assert oracle.fp4_block_exponent(a) == exact_exponent(a), a
    # away from the clamp it is ceil(log2(amax / 6)): exact at the powers 6 * 2^k
    for k in range(-20, 21):
        assert oracle.fp4_block_exponent(6.0 * 2.0**k) == k
        assert oracle.fp4_block_exponent(np.nextafter(6.0 * 2.0**k, np.inf)) == k + 1


def row_bits(vals, d):
    x = np.zeros(d, np.float32)
    x[: len(vals)] = vals
    return bits(torch.tensor(x).to(torch.bfloat16)).reshape(1, 1, 1, d)


def test_quantize_row_by_hand(oracle):
    # block 0: amax 6 -> e = 0 (scale byte 127); 6 -> 7, -3 -> 8|5 = 13, 1.5 -> 3, 0.703125 -> 1 (0.5),
    #          0.25 -> 0 (tie to even), 0 -> 0;  bytes (lo | hi << 4): 0xD7, 0x13, 0x00
    # block 1: amax 0.30078125 -> e = -4 (6/16 = 0.375 >= amax > 6/32), scale byte 123;
    #          0.30078125 * 16 = 4.8125 -> 4 (code 6), -0.0625 * 16 = -1 -> code 10
    d = 64
    x = np.zeros(d, np.float32)
    x[:6] = [6.0, -3.0, 1.5, 0.703125, 0.25, 0.0]
    x[32], x[33] = 0.30078125, -0.0625
    codes, sc = oracle.quantize_kv_fp4(bits(torch.tensor(x).to(torch.bfloat16)).reshape(1, 1, 1, d))
    assert list(sc.ravel()) == [127, 123]
    c = codes.ravel()
    assert list(c[:3]) == [0xD7, 0x13, 0x00] and not c[3:16].any()
    assert c[16] == (6 | (10 << 4)) and not c[17:].any()
    # an all-zero row: exponent -126 (scale byte 1), zero codes
    codes, sc = oracle.quantize_kv_fp4(row_bits([], 32))
    assert list(sc.ravel()) == [1] and not codes.any()


def grid_cache(rng, B, H, L, d):
    """Rows whose every 32-channel block holds e2m1 values times 2^e with one
    entry of magnitude exactly 6 * 2^e: their encoding is exact."""
    nb = d // 32
    c = rng.integers(0, 16, size=(B, H, L, d)).astype(np.uint8)
    c.reshape(B, H, L, nb, 32)[..., 0] = np.where(rng.integers(0, 2, size=(B, H, L, nb)) == 1, 7, 15)
    e = rng.integers(-10, 10, size=(B, H, L, nb))
    table = np.array(E2M1 + [-v for v in E2M1])
    vals = table[c].reshape(B, H, L, nb, 32) * np.exp2(e)[..., None]
    vals = vals.reshape(B, H, L, d)
    x = bits(torch.tensor(vals).to(torch.bfloat16))
    assert np.array_equal((x.astype(np.uint32) << 16).view(np.float32).astype(np.float64), vals)
    packed = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    # -0 (code 8) encodes as +0's sign-preserving code 8 only if the value is -0.0; bf16 keeps -0
    return x, packed, (e + 127).astype(np.uint8)


def test_exact_round_trip(oracle):
    rng = np.random.default_rng(13)
    x, c, s = grid_cache(rng, 2, 3, 40, 128)
    codes, sc = oracle.quantize_kv_fp4(x)
    np.testing.assert_array_equal(sc, s)
    np.testing.assert_array_equal(codes, c)
    deq = oracle.dequantize_kv_fp4(codes, sc)
    np.testing.assert_array_equal(deq, (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


def test_error_bound(oracle):
    rng = np.random.default_rng(14)
    B, H, L, d = 2, 2, 50, 128
    mag = np.exp2(rng.uniform(-30, 30, size=(B, H, L, 1)))
    xf = rng.standard_normal((B, H, L, d)) * mag
    x = bits(torch.tensor(xf, dtype=torch.float32).to(torch.bfloat16))
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, sc = oracle.quantize_kv_fp4(x)
    deq = oracle.dequantize_kv_fp4(codes, sc)
    step = np.exp2(sc.astype(np.float64) - 127)  # 2^e per block
    step = np.repeat(step, 32, axis=-1)
    # half the largest e2m1 spacing (2, between 4 and 6), in units of 2^e; and the
    # spacing is at most 1/4 of |x| once |x| * 2^-e >= 1
    assert np.all(np.abs(deq - xv) <= step)
    big = np.abs(xv) >= step
    assert np.all(np.abs(deq - xv)[big] <= 0.25 * np.abs(xv)[big])
    assert np.all((np.sign(deq) == np.sign(xv)) | (deq == 0))
    # e is minimal, so each block's max |x| * 2^-e lies in (3, 6] and decodes to 3, 4 or 6
    blk = np.abs(deq).reshape(B, H, L, d // 32, 32).max(axis=-1) / np.exp2(sc.astype(np.float64) - 127)
    assert np.all(np.isin(blk, [3.0, 4.0, 6.0]))


def test_rows_past_seq_len_untouched(oracle):
    x = bits(torch.randn(2, 2, 30, 64).to(torch.bfloat16))
    sl = np.array([17, 0], np.int32)
    codes, sc = oracle.quantize_kv_fp4(x, sl)
    assert not codes[0, :, 17:].any() and not sc[0, :, 17:].any() and not codes[1].any() and not sc[1].any()
    full, fsc = oracle.quantize_kv_fp4(x)
    np.testing.assert_array_equal(codes[0, :, :17], full[0, :, :17])
    np.testing.assert_array_equal(sc[0, :, :17], fsc[0, :, :17])


def test_fp4_attention_reduces_to_bf16_when_exact(oracle):
    rng = np.random.default_rng(15)
    B, Hq, Hkv, L, d = 2, 4, 2, 70, 64
    k, kc, ks = grid_cache(rng, B, Hkv, L, d)
    v, vc, vs = grid_cache(rng, B, Hkv, L, d)
    q = bits(torch.randn(B, Hq, d).to(torch.bfloat16))
    sl = np.array([70, 33], np.int32)
    out4, lse4 = oracle.decode_dense_fp4(q, kc, ks, oracle.fp4_rows_to_pairs(vc, sl), vs, sl, 0.02)
    out, lse = oracle.decode_dense(q, k, v, sl, 0.02)
    np.testing.assert_allclose(out4, out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse4, lse, rtol=1e-13, atol=1e-13)


# ------------------------------------------------- value cache in token pairs

def test_value_pairs_by_hand(oracle):
    # two rows of d = 64: channel c of row 0 has code c % 16, of row 1 code (c + 5) % 16
    c0 = np.arange(64) % 16
    c1 = (np.arange(64) + 5) % 16
    rows = np.stack([c0, c1]).astype(np.uint8)                    # [2, 64] codes
    keylayout = (rows[:, 0::2] | (rows[:, 1::2] << 4)).reshape(1, 1, 2, 32)
    pairs = oracle.fp4_rows_to_pairs(keylayout)
    assert pairs.shape == (1, 1, 1, 64)
    np.testing.assert_array_equal(pairs[0, 0, 0], (c1 << 4) | c0)  # low nibble: the even token
    np.testing.assert_array_equal(oracle.fp4_pairs_to_rows(pairs, 2), keylayout)


def test_value_pairs_odd_length_and_seq_lens(oracle):
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(2, 3, 7, 32)).astype(np.uint8)   # L = 7 (odd)
    sl = np.array([7, 4], np.int32)
    pairs = oracle.fp4_rows_to_pairs(codes, sl)
    assert pairs.shape == (2, 3, 4, 64)
    # the last pair of a 7-token sequence holds token 6 and code 0 for the absent token 7
    assert not (pairs[0, :, 3] >> 4).any()
    np.testing.assert_array_equal(oracle.fp4_pairs_to_rows(pairs, 7)[0], codes[0])
    # sequence 1 has 4 tokens: pairs 2, 3 stay zero, the first two round-trip
    assert not pairs[1, :, 2:].any()
    np.testing.assert_array_equal(oracle.fp4_pairs_to_rows(pairs, 7)[1, :, :4], codes[1, :, :4])


def test_value_pair_encoding_decodes_like_the_key_layout(oracle):
    x = bits(torch.randn(2, 2, 45, 128).to(torch.bfloat16))
    sl = np.array([45, 20], np.int32)
    kc, ks = oracle.quantize_kv_fp4(x, sl)
    vc, vs = oracle.quantize_v_fp4(x, sl)
    np.testing.assert_array_equal(vs, ks)
    np.testing.assert_array_equal(oracle.dequantize_v_fp4(vc, vs, sl), oracle.dequantize_kv_fp4(kc, ks, sl))
