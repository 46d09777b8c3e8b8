"""Pins for the oracle's key encoder and its FFD top-delta decode.

The encoder is this library's own definition (the FFD summary, section 5,
names a 2-bit body plus an 8-bit residual but gives no formulas), so it is
pinned by hand-derived groups (expected bits worked out in the comments),
by the IEEE binary16 conversion of numpy, and by its error bounds.  The
top-delta decode is pinned by hand-built score profiles whose pseudo-max,
candidate set and output follow in closed form, by its reduction to dense
attention at delta = +inf, and by the invariants of the rule s~ >= m^ - delta.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return bits(t)


def encode_group(oracle, x32):
    """Encode one 32-channel group given as python floats (exact in bf16)."""
    k = bf16_bits_of(x32).reshape(1, 1, 1, 32)
    return oracle.quantize_keys(k)


# ------------------------------------------------------------ binary16 rounding

def test_float_to_half_matches_numpy(oracle):
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-27, 17, 20000)).astype(np.float32)
    x = np.concatenate([mags * rng.choice([-1.0, 1.0], mags.size).astype(np.float32),
                        np.array([0.0, -0.0, 1.0 + 2**-11, 1.0 + 3 * 2**-11, 65504.0, 65519.99,
                                  65520.0, 1e6, 2**-24, 2**-25, 3 * 2**-26, 2**-14 - 2**-25,
                                  5.9604645e-08, np.inf, -np.inf], np.float32)])
    ours = oracle.float_to_half(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = oracle.half_to_float(ref)
    np.testing.assert_array_equal(back, ref.view(np.float16).astype(np.float32))


# ---------------------------------------------------------- hand-derived groups

def test_encode_grid_group(oracle):
    # x = [-1, 0, 1, 2] * 8: mn = -1, mx = 2, (mx - mn)/3 = 1 -> s16 = 1.0 (0x3C00),
    # mn16 = -1.0 (0xBC00); codes (x + 1)/1 = 0,1,2,3 -> each byte 0|1<<2|2<<4|3<<6 = 0xE4;
    # deq2 == x, residual 0 -> rs16 = 0, rq = 0.
    codes, ms, res, rs = encode_group(oracle, [-1.0, 0.0, 1.0, 2.0] * 8)
    assert list(codes.ravel()) == [0xE4] * 8
    assert list(ms.ravel()) == [0xBC00, 0x3C00]
    assert not res.any() and rs.ravel()[0] == 0


def test_encode_constant_group(oracle):
    # all 0.75: mx - mn = 0 -> s16 = 0, every code 0, mn16 = 0.75 = 0x3A00, residual 0
    codes, ms, res, rs = encode_group(oracle, [0.75] * 32)
    assert not codes.any()
    assert list(ms.ravel()) == [0x3A00, 0x0000]
    assert not res.any() and rs.ravel()[0] == 0


def test_encode_rounded_scale_group(oracle):
    # x = [0.5, 1.25, 0 * 30]: mn = 0, mx = 1.25.
    #  (mx-mn)/3 in binary32 = 0.41666666...; binary16 spacing on [0.25, 0.5) is 2^-12,
    #  0.41666/2^-12 = 1706.67 -> 1707 * 2^-12 = 0.416748046875 = 0x36AB.
    #  codes: 0.5/0.41675 = 1.1998 -> 1; 1.25/0.41675 = 2.9994 -> 3; zeros -> 0;
    #  byte 0 = 1 | 3<<2 = 0x0D.
    #  deq2 = 0.416748046875, 1.250244140625; r = 0.083251953125 (= 341 * 2^-12), -2^-12.
    #  max|r|/127 = 341*2^-12/127; on [2^-11, 2^-10) the spacing is 2^-21:
    #  341 * 2^9 / 127 = 1374.74 -> 1375 * 2^-21 = 0x115F.
    #  rq: 341*2^9/1375 = 126.98 -> 127;  -2^-12 / (1375*2^-21) = -0.372 -> 0.
    x = [0.5, 1.25] + [0.0] * 30
    codes, ms, res, rs = encode_group(oracle, x)
    assert list(codes.ravel()) == [0x0D] + [0] * 7
    assert list(ms.ravel()) == [0x0000, 0x36AB]
    assert list(res.ravel()) == [127] + [0] * 31
    assert list(rs.ravel()) == [0x115F]


def test_encode_ties_round_to_even(oracle):
    # x = [0, 3, 0.5, 1.5, 2.5, 0 * 27]: mn = 0, s16 = 1.0.
    #  ratios 0, 3, 0.5, 1.5, 2.5 -> rint to even: 0, 3, 0, 2, 2.
    #  byte 0 = 0 | 3<<2 | 0<<4 | 2<<6 = 0x8C; byte 1 = 2 = 0x02.
    #  r = 0, 0, 0.5, -0.5, 0.5; max|r|/127 = 0.5/127 = 0.0039370; on [2^-8, 2^-7) the
    #  spacing is 2^-18: 2^17/127 = 1032.06 -> 1032 * 2^-18 = 0x1C08.
    #  rq = +-0.5/(1032*2^-18) = +-127.008 -> clamp to +-127.
    x = [0.0, 3.0, 0.5, 1.5, 2.5] + [0.0] * 27
    codes, ms, res, rs = encode_group(oracle, x)
    assert list(codes.ravel()) == [0x8C, 0x02] + [0] * 6
    assert list(ms.ravel()) == [0x0000, 0x3C00]
    assert list(res.ravel()) == [0, 0, 127, -127, 127] + [0] * 27
    assert list(rs.ravel()) == [0x1C08]


@pytest.mark.parametrize("x", [[-0.0] * 32, [-0.0, 0.0] * 16, [0.0, -0.0] * 16])
def test_encode_signed_zero_group(oracle, x):
    # a zero extreme is +0 whatever its sign: mn16 = +0 (0x0000), s16 = +0, codes 0, residual 0
    codes, ms, res, rs = encode_group(oracle, x)
    assert list(ms.ravel()) == [0x0000, 0x0000]
    assert not codes.any() and not res.any() and rs.ravel()[0] == 0


def test_encoder_leaves_rows_past_the_end(oracle):
    p = W.random_problem(2, 2, 2, 40, 64, seed=1, seq_lens=[40, 7])
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k), p.seq_lens)
    assert not codes[1, :, 7:].any() and not res[1, :, 7:].any()
    assert not ms[1, :, 7:].any() and not rs[1, :, 7:].any()
    full = oracle.quantize_keys(bits(p.k[1:2, :, :7]))
    np.testing.assert_array_equal(codes[1, :, :7], full[0][0])
    np.testing.assert_array_equal(res[1, :, :7], full[2][0])


# ------------------------------------------------------------- error bounds

@pytest.mark.parametrize("std", [1.0, 1e-3, 40.0])
def test_encoder_error_bounds(oracle, std):
    p = W.random_problem(1, 2, 2, 300, 128, seed=3, std=std)
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k))
    x = p.k.double().numpy()
    d2 = oracle.dequantize_keys(codes, ms, res, rs, with_residual=False)
    kt = oracle.dequantize_keys(codes, ms, res, rs, with_residual=True)
    mn = oracle.half_to_float(ms[..., 0]).astype(np.float64).reshape(ms.shape[:-1])
    s = oracle.half_to_float(ms[..., 1]).astype(np.float64).reshape(ms.shape[:-1])
    rsf = oracle.half_to_float(rs).astype(np.float64).reshape(rs.shape)
    xg = x.reshape(*x.shape[:-1], 4, 32)
    # codes are 2-bit, residuals within the symmetric int8 range
    assert res.min() >= -127 and res.max() <= 127
    # 2-bit body: within half a step of x, unless x lies beyond the top of the
    # (rounded) grid, where the top code is taken
    top = mn + 3 * s
    over = np.maximum(xg.max(-1) - top, 0.0)
    err2 = np.abs(xg - d2.reshape(xg.shape)).max(-1)
    tol = 1e-6 * (np.abs(xg).max(-1) + 1e-30)
    assert np.all(err2 <= np.maximum(s / 2, over) + np.abs(mn - xg.min(-1)) + tol)
    # residual-corrected key: within half a residual step, unless max|r| lies past 127 steps
    r = xg - d2.reshape(xg.shape)
    amax = np.abs(r).max(-1)
    clip = np.maximum(amax - 127 * rsf, 0.0)
    errk = np.abs(xg - kt.reshape(xg.shape)).max(-1)
    assert np.all(errk <= np.maximum(rsf / 2, clip) + tol)
    # the residual refines: never worse than the 2-bit body alone
    assert np.all(errk <= err2 + tol)


# ------------------------------------------------------ top-delta: hand profiles

def crafted(mn_values, d=32, res_q=None, res_scale=None, v=None):
    """Quantized keys whose 2-bit body is the constant mn_t on every channel
    (s16 = 0, all codes 0), so with q = 1/d on every channel and scale 1 the
    2-bit score is exactly s~_t = mn_t.  Optional residual rq (per token, all
    channels) with scale rs16 per token."""
    L = len(mn_values)
    ng = d // 32
    codes = np.zeros((1, 1, L, d // 4), np.uint8)
    ms = np.zeros((1, 1, L, ng, 2), np.uint16)
    ms[..., 0] = np.asarray(mn_values, np.float16).view(np.uint16)[None, None, :, None]
    res = np.zeros((1, 1, L, d), np.int8)
    rs = np.zeros((1, 1, L, ng), np.uint16)
    if res_q is not None:
        res[0, 0] = np.asarray(res_q, np.int8)[:, None]
        rs[0, 0] = np.asarray(res_scale, np.float16).view(np.uint16)[:, None]
    q = torch.full((1, 1, d), 1.0 / d).to(torch.bfloat16)
    if v is None:
        v = torch.randn((1, 1, L, d), generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    return q, codes, ms, res, rs, v


def test_pseudo_max_uses_only_sinks_and_window(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    # L = 200, 4 sinks, window 64: anchors {0..3} U {136..199}.
    mn = np.full(200, -8.0)
    mn[2] = 1.0        # sink
    mn[136] = 1.5      # first token of the window: the pseudo-max
    mn[150] = 1.25     # window
    mn[100] = 4.0      # true maximum, not an anchor
    mn[4] = 3.0        # first token after the sinks (not an anchor)
    mn[135] = 3.0      # last token before the window (not an anchor)
    mn[50] = -3.5      # exactly m^ - delta: kept (inclusive)
    mn[51] = -3.50390625  # one binary16 step below: dropped
    q, codes, ms, res, rs, v = crafted(mn)
    r = oracle.decode_topdelta(q, codes, ms, res, rs, v, None, 1.0, 5.0, n_sink=4, window=64,
                               want_scores=True)
    assert r["m_hat"][0, 0] == 1.5
    np.testing.assert_array_equal(r["s_tilde"][0, 0], mn)
    sel = [j for j in range(200) if (r["sel_mask"][0, 0, j // 32] >> (j % 32)) & 1]
    assert sel == [2, 4, 50, 100, 135, 136, 150]
    assert r["sel_count"][0, 0] == 7
    s = mn[sel]
    w = scipy_special.softmax(s)
    np.testing.assert_allclose(r["out"][0, 0], w @ v[0, 0, sel].double().numpy(), atol=1e-13)
    assert r["lse"][0, 0] == pytest.approx(scipy_special.logsumexp(s), abs=1e-13)


def test_selection_on_2bit_scores_attention_on_corrected_scores(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    # anchors give m^ = 0 (tokens 0..3 and the window all at 0, L = 80 -> window 16..79).
    # token 5: s~ = -6 (dropped at delta=5) although its corrected score
    #          -6 + 127/32 = -2.03125 would pass; token 9: s~ = -3 (kept) with corrected
    #          score -3 - 127/32 = -6.96875, which is the score its weight uses.
    L = 80
    mn = np.full(L, -20.0)
    mn[:4] = 0.0
    mn[16:] = 0.0
    mn[5] = -6.0
    mn[9] = -3.0
    rq = np.zeros(L, np.int8)
    rsc = np.zeros(L, np.float32)
    rq[5], rsc[5] = 127, 1.0 / 32
    rq[9], rsc[9] = -127, 1.0 / 32
    q, codes, ms, res, rs, v = crafted(mn, res_q=rq, res_scale=rsc)
    r = oracle.decode_topdelta(q, codes, ms, res, rs, v, None, 1.0, 5.0, n_sink=4, window=64)
    sel = [j for j in range(L) if (r["sel_mask"][0, 0, j // 32] >> (j % 32)) & 1]
    expect = list(range(4)) + [9] + list(range(16, L))
    assert sel == expect
    s = np.zeros(len(expect))
    s[expect.index(9)] = -3.0 - 127.0 / 32
    w = scipy_special.softmax(s)
    np.testing.assert_allclose(r["out"][0, 0], w @ v[0, 0, expect].double().numpy(), atol=1e-13)
    assert r["lse"][0, 0] == pytest.approx(scipy_special.logsumexp(s), abs=1e-13)


def test_single_candidate_returns_its_value(oracle):
    # only the anchor at the pseudo-max passes a delta of 0: out = v_j, LSE = s_j
    mn = np.full(70, -1.0)
    mn[3] = 2.0
    q, codes, ms, res, rs, v = crafted(mn)
    # move the window away from token 3: L = 70 -> window = {6..69}
    r = oracle.decode_topdelta(q, codes, ms, res, rs, v, None, 1.0, 0.0, n_sink=4, window=64)
    assert r["sel_count"][0, 0] == 1 and r["sel_mask"][0, 0, 0] == (1 << 3)
    np.testing.assert_array_equal(r["out"][0, 0], v[0, 0, 3].double().numpy())
    assert r["lse"][0, 0] == 2.0


def test_empty_and_short_sequences(oracle):
    p = W.random_problem(3, 4, 2, 50, 64, seed=5, seq_lens=[0, 3, 50])
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k), p.seq_lens)
    r = oracle.decode_topdelta(bits(p.q), codes, ms, res, rs, bits(p.v), p.seq_lens, p.scale, 5.0)
    assert np.all(r["out"][0] == 0) and np.all(np.isneginf(r["lse"][0]))
    assert np.all(r["sel_count"][0] == 0) and not r["sel_mask"][0].any()
    # L = 3 < n_sink: every token is an anchor, so the anchor maximum is the global one
    assert np.all(r["sel_count"][1] >= 1)


# ----------------------------------------------------------- reductions, laws

def ffd_small(seed=0, B=2, L=700, Hq=8, Hkv=2, d=128):
    return W.ffd(seed=seed, B=B, L=L, Hq=Hq, Hkv=Hkv, d=d)


def test_infinite_delta_is_dense_attention_on_dequantized_keys(oracle):
    p = ffd_small(seed=7)
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k))
    r = oracle.decode_topdelta(bits(p.q), codes, ms, res, rs, bits(p.v), None, p.scale, math.inf)
    assert np.all(r["sel_count"] == p.L_max)
    kt = oracle.dequantize_keys(codes, ms, res, rs)
    ref, lref = oracle.decode_dense_f64(p.q.double().numpy(), kt, p.v.double().numpy(), None, p.scale)
    np.testing.assert_allclose(r["out"], ref, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lref, atol=1e-12)
    # and close to dense attention on the bf16 keys: the encoder error bounds the gap
    dense, ldense = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    kerr = np.abs(kt - p.k.double().numpy()).max()
    qn1 = np.abs(p.q.double().numpy()).sum(-1).max()
    ds = p.scale * qn1 * kerr
    assert np.abs(r["lse"] - ldense).max() <= ds + 1e-12
    assert np.abs(r["out"] - dense).max() <= 2 * ds * np.abs(p.v.double().numpy()).max() + 1e-12


def test_rule_laws(oracle):
    p = ffd_small(seed=9, L=1000)
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k))
    r5 = oracle.decode_topdelta(bits(p.q), codes, ms, res, rs, bits(p.v), None, p.scale, 5.0,
                                want_scores=True)
    r7 = oracle.decode_topdelta(bits(p.q), codes, ms, res, rs, bits(p.v), None, p.scale, 7.0)
    # nested: delta = 5 keeps a subset of delta = 7
    assert np.all((r5["sel_mask"] & ~r7["sel_mask"]) == 0)
    assert np.all(r5["sel_count"] <= r7["sel_count"])
    # s~ is the score on the 2-bit body (cross-checked through the dequantizer)
    d2 = oracle.dequantize_keys(codes, ms, res, rs, with_residual=False)
    G = p.Hq // p.Hkv
    qd = p.q.double().numpy()
    L = p.L_max
    for b in range(p.B):
        for hq in range(p.Hq):
            st = p.scale * (d2[b, hq // G] @ qd[b, hq])
            np.testing.assert_allclose(r5["s_tilde"][b, hq], st, atol=1e-12)
            anchors = np.r_[0:4, L - 64:L]
            assert r5["m_hat"][b, hq] == st[anchors].max()
            mask = np.array([(r5["sel_mask"][b, hq, j // 32] >> (j % 32)) & 1 for j in range(L)], bool)
            np.testing.assert_array_equal(mask, st >= st[anchors].max() - 5.0)
            # the anchor that sets the pseudo-max is always a candidate
            assert mask[anchors[np.argmax(st[anchors])]]


# ------------------------------------------- candidate set shared by a KV group

def two_head_profiles(mn0, mn1):
    """Two query heads on one KV head, d = 64: head 0 reads only channels
    0..31 (q = 1/32 there), head 1 only channels 32..63, and the 2-bit body of
    token t is the constant mn0[t] on the first group and mn1[t] on the
    second (s16 = 0), so with scale 1 head g's 2-bit score is mn_g[t]."""
    L = len(mn0)
    d = 64
    codes = np.zeros((1, 1, L, d // 4), np.uint8)
    ms = np.zeros((1, 1, L, 2, 2), np.uint16)
    ms[0, 0, :, 0, 0] = np.asarray(mn0, np.float16).view(np.uint16)
    ms[0, 0, :, 1, 0] = np.asarray(mn1, np.float16).view(np.uint16)
    res = np.zeros((1, 1, L, d), np.int8)
    rs = np.zeros((1, 1, L, 2), np.uint16)
    q = torch.zeros((1, 2, d))
    q[0, 0, :32] = 1.0 / 32
    q[0, 1, 32:] = 1.0 / 32
    q = q.to(torch.bfloat16)
    v = torch.randn((1, 1, L, d), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    return q, codes, ms, res, rs, v


def test_group_union_hand_profile(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    # L = 100, 4 sinks, window 64 -> anchors {0..3} U {36..99}, all at 0 for both heads: m^ = 0.
    # Token 10: head 0 scores -2 (kept at delta 5), head 1 scores -9 (dropped).
    # Token 20: head 0 scores -8 (dropped), head 1 scores -1 (kept).  Other tokens -20.
    L = 100
    mn0 = np.full(L, -20.0)
    mn1 = np.full(L, -20.0)
    for mn in (mn0, mn1):
        mn[:4] = 0.0
        mn[36:] = 0.0
    mn0[10], mn1[10] = -2.0, -9.0
    mn0[20], mn1[20] = -8.0, -1.0
    q, codes, ms, res, rs, v = two_head_profiles(mn0, mn1)
    r = oracle.decode_topdelta_group_union(q, codes, ms, res, rs, v, None, 1.0, 5.0, 4, 64)
    anchors = list(range(4)) + list(range(36, L))
    own = {0: sorted(anchors + [10]), 1: sorted(anchors + [20])}
    union = sorted(anchors + [10, 20])
    for g, mn in ((0, mn0), (1, mn1)):
        got_own = [j for j in range(L) if (r["head_sel_mask"][0, g, j // 32] >> (j % 32)) & 1]
        got = [j for j in range(L) if (r["sel_mask"][0, g, j // 32] >> (j % 32)) & 1]
        assert got_own == own[g] and got == union
        assert r["sel_count"][0, g] == len(union) and r["head_sel_count"][0, g] == len(own[g])
        # every head weighs the whole union with its own scores
        s = mn[union]
        w = scipy_special.softmax(s)
        np.testing.assert_allclose(r["out"][0, g], w @ v[0, 0, union].double().numpy(), atol=1e-13)
        assert r["lse"][0, g] == pytest.approx(scipy_special.logsumexp(s), abs=1e-13)


def test_group_union_laws(oracle):
    p = ffd_small(seed=11, L=900)
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k))
    args = (bits(p.q), codes, ms, res, rs, bits(p.v), None, p.scale)
    G = p.Hq // p.Hkv
    for delta in (2.0, 5.0):
        per = oracle.decode_topdelta(*args, delta)
        uni = oracle.decode_topdelta_group_union(*args, delta)
        np.testing.assert_array_equal(uni["head_sel_mask"], per["sel_mask"])
        grp = uni["sel_mask"].reshape(p.B, p.Hkv, G, -1)
        # the union contains every head's set and is the same for the whole group
        assert np.all((per["sel_mask"] & ~uni["sel_mask"]) == 0)
        assert np.all(grp == grp[:, :, :1])
        # attending to more keys can only raise log sum exp
        assert np.all(uni["lse"] >= per["lse"] - 1e-12)
    # delta = inf: everything is selected and the result is dense attention on k~
    uni = oracle.decode_topdelta_group_union(*args, math.inf)
    kt = oracle.dequantize_keys(codes, ms, res, rs)
    ref, lref = oracle.decode_dense_f64(p.q.double().numpy(), kt, p.v.double().numpy(), None, p.scale)
    np.testing.assert_allclose(uni["out"], ref, atol=1e-12)
    np.testing.assert_allclose(uni["lse"], lref, atol=1e-12)


def test_group_union_of_one_head_is_the_per_head_rule(oracle):
    p = W.ffd(seed=12, B=2, L=700, Hq=4, Hkv=4, d=64)
    lens = torch.tensor([700, 333], dtype=torch.int32)
    codes, ms, res, rs = oracle.quantize_keys(bits(p.k), lens)
    args = (bits(p.q), codes, ms, res, rs, bits(p.v), lens, p.scale, 5.0)
    per = oracle.decode_topdelta(*args)
    uni = oracle.decode_topdelta_group_union(*args)
    np.testing.assert_array_equal(uni["sel_mask"], per["sel_mask"])
    np.testing.assert_array_equal(uni["sel_count"], per["sel_count"])
    np.testing.assert_allclose(uni["out"], per["out"], atol=1e-12)
    np.testing.assert_allclose(uni["lse"], per["lse"], atol=1e-12)
