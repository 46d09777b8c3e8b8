"""Pins for the oracle's dense, split and paged decode attention.

Each test ties the oracle to something other than itself: a closed form, a
library routine (scipy's softmax / logsumexp, torch's scaled-dot-product
attention in float64), high-precision brute force on tiny integer inputs, or
an invariance the method guarantees ("Flash Decoding" tutorial, section 2 and
the misconceptions section: split + merge is an identity).  The page's numpy
demo fixes only its shape (no value is printed), kept in tests/golden.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t):
    return t.double().numpy()


def small(B=2, Hq=4, Hkv=2, L=50, d=16, seed=0, seq_lens=None):
    return W.random_problem(B, Hq, Hkv, L, d, seed=seed, seq_lens=seq_lens)


# ---------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_values(oracle):
    # all keys equal => every weight is 1/L: out = mean_j v_j, LSE = s + ln L
    B, Hq, Hkv, L, d = 1, 3, 1, 37, 8
    p = W.random_problem(B, Hq, Hkv, L, d, seed=3)
    k = p.k.clone()
    k[:] = k[:, :, :1, :]
    out, lse = oracle.decode_dense(bits(p.q), bits(k), bits(p.v), None, p.scale)
    V = f64(p.v)[0, 0]
    np.testing.assert_allclose(out[0], np.broadcast_to(V.mean(axis=0), (Hq, d)), rtol=0, atol=1e-13)
    s = p.scale * (f64(p.q)[0] @ f64(k)[0, 0, 0])
    np.testing.assert_allclose(lse[0], s + math.log(L), rtol=0, atol=1e-12)


def test_one_dominant_key_returns_its_value(oracle):
    # key j* = k + c*q_hat with a score gap of >= 40 over every other key:
    # out = v_j* up to sum_{j != j*} e^{-40} |v_j|, LSE = s_j* up to L e^{-40}
    B, Hq, Hkv, L, d = 1, 1, 1, 64, 16
    p = W.random_problem(B, Hq, Hkv, L, d, seed=5)
    q = f64(p.q)[0, 0]
    K = f64(p.k)[0, 0].copy()
    jstar = 41
    qn = q / np.linalg.norm(q)
    K[jstar] += (45.0 / p.scale / np.linalg.norm(q)) * qn
    s = p.scale * (K @ q)
    gap = s[jstar] - np.max(np.delete(s, jstar))
    assert gap >= 40
    out, lse = oracle.decode_dense_f64(q[None, None], K[None, None], f64(p.v), None, p.scale)
    V = f64(p.v)[0, 0]
    np.testing.assert_allclose(out[0, 0], V[jstar], rtol=0, atol=L * math.exp(-40) * np.abs(V).max())
    assert abs(lse[0, 0] - s[jstar]) <= L * math.exp(-40) + 1e-14 * abs(s[jstar])


def test_gqa_head_mapping(oracle):
    # query head hq reads KV head hq // G: give every KV head a constant value
    # row equal to its index, so out[hq] = hq // G exactly.
    B, Hq, Hkv, L, d = 2, 8, 2, 19, 8
    p = W.random_problem(B, Hq, Hkv, L, d, seed=7)
    v = torch.zeros_like(p.v)
    for h in range(Hkv):
        v[:, h] = float(h + 1)
    out, _ = oracle.decode_dense(bits(p.q), bits(p.k), bits(v), None, p.scale)
    G = Hq // Hkv
    for hq in range(Hq):
        np.testing.assert_allclose(out[:, hq], hq // G + 1.0, rtol=0, atol=1e-13)


def test_empty_sequence(oracle):
    p = small(B=3, seq_lens=[5, 0, 50])
    out, lse = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens, p.scale)
    assert np.all(out[1] == 0.0)
    assert np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[0])) and np.all(np.isfinite(lse[2]))


def test_seq_lens_ignore_tokens_past_the_end(oracle):
    # tokens at t >= L_b must not contribute: poison them with huge keys
    p = small(B=2, L=40, seq_lens=[17, 40])
    k = p.k.clone()
    k[0, :, 17:] = 300.0
    a, la = oracle.decode_dense(bits(p.q), bits(k), bits(p.v), p.seq_lens, p.scale)
    b_, lb = oracle.decode_dense(bits(p.q[:1]), bits(p.k[:1, :, :17]), bits(p.v[:1, :, :17]), None, p.scale)
    np.testing.assert_array_equal(a[0], b_[0])
    np.testing.assert_array_equal(la[0], lb[0])


# ---------------------------------------------------------- library routines

def test_matches_scipy_softmax(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    p = small(B=2, Hq=6, Hkv=3, L=77, d=32, seed=11, seq_lens=[77, 30])
    out, lse = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens, p.scale)
    q, K, V = f64(p.q), f64(p.k), f64(p.v)
    G = p.Hq // p.Hkv
    for b in range(p.B):
        L = int(p.seq_lens[b])
        for hq in range(p.Hq):
            s = p.scale * (K[b, hq // G, :L] @ q[b, hq])
            w = scipy_special.softmax(s)
            np.testing.assert_allclose(out[b, hq], w @ V[b, hq // G, :L], rtol=1e-12, atol=1e-13)
            assert abs(lse[b, hq] - scipy_special.logsumexp(s)) < 1e-12


def test_matches_torch_sdpa_float64(oracle):
    p = small(B=2, Hq=8, Hkv=2, L=129, d=64, seed=13)
    out, lse = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    q = p.q.double()[:, :, None, :]          # [B, Hq, 1, d]
    G = p.Hq // p.Hkv
    k = p.k.double().repeat_interleave(G, dim=1)
    v = p.v.double().repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=p.scale)[:, :, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_integer_brute_force_high_precision(oracle):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(2024)
    for L in range(1, 9):
        d = 4
        q = rng.integers(-3, 4, size=d).astype(np.float64)
        K = rng.integers(-3, 4, size=(L, d)).astype(np.float64)
        V = rng.integers(-5, 6, size=(L, d)).astype(np.float64)
        scale = 0.5
        out, lse = oracle.decode_dense_f64(q[None, None], K[None, None], V[None, None], None, scale)
        s = [mpmath.mpf(scale) * sum(mpmath.mpf(q[c]) * mpmath.mpf(K[j, c]) for c in range(d))
             for j in range(L)]
        e = [mpmath.e ** x for x in s]
        Z = sum(e)
        for c in range(d):
            ref = sum(e[j] * mpmath.mpf(V[j, c]) for j in range(L)) / Z
            assert abs(out[0, 0, c] - float(ref)) <= 1e-14 * (1 + abs(float(ref)))
        assert abs(lse[0, 0] - float(mpmath.log(Z))) <= 1e-14 * (1 + abs(float(mpmath.log(Z))))


# ---------------------------------------------------------------- split form

@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 50, 64])
def test_split_merge_is_exact(oracle, S):
    # the tutorial's claim: chunked statistics + the max merge reproduce
    # standard attention (up to rounding) for any number of chunks
    p = small(B=2, Hq=4, Hkv=2, L=50, d=16, seed=17, seq_lens=[50, 23])
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens, p.scale)
    out, lse, pm, pl, po = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), p.seq_lens, p.scale, S)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-12)


def test_split_one_token_per_chunk_closed_form(oracle):
    # with one token per chunk: m_i = s_i, l_i = 1 and the normalised O_i = v_i
    p = small(B=1, Hq=2, Hkv=1, L=9, d=8, seed=19)
    out, lse, pm, pl, po = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), None, p.scale, 9)
    s = p.scale * np.einsum("hd,ld->hl", f64(p.q)[0], f64(p.k)[0, 0])
    np.testing.assert_allclose(pm[0], s, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(pl[0], 1.0)
    for h in range(2):
        np.testing.assert_array_equal(po[0, h], f64(p.v)[0, 0])


def test_split_chunks_cover_every_token_and_empty_chunks(oracle):
    # L=10, S=4: chunk size ceil(10/4)=3 -> chunks [0,3) [3,6) [6,9) [9,10);
    # L=10, S=7: size 2 -> chunks 0..4 hold 2 tokens each, chunks 5, 6 are empty
    p = small(B=1, Hq=1, Hkv=1, L=10, d=8, seed=23)
    _, _, pm, pl, _ = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), None, p.scale, 4)
    s = p.scale * (f64(p.k)[0, 0] @ f64(p.q)[0, 0])
    for i, (a, b) in enumerate([(0, 3), (3, 6), (6, 9), (9, 10)]):
        assert pm[0, 0, i] == pytest.approx(s[a:b].max(), abs=1e-13)
        assert pl[0, 0, i] == pytest.approx(np.exp(s[a:b] - s[a:b].max()).sum(), abs=1e-13)
    _, _, pm, pl, _ = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), None, p.scale, 7)
    assert np.all(np.isneginf(pm[0, 0, 5:])) and np.all(pl[0, 0, 5:] == 0)
    assert np.all(np.isfinite(pm[0, 0, :5]))


def test_as_printed_unnormalised_merge_is_wrong(oracle):
    # Reading taken for the tutorial's inconsistent step 1: the merge multiplies
    # O_i by l_i, so O_i must be the locally normalised output.  Using the
    # un-normalised sum there (as the demo listing does) breaks exactness.
    p = small(B=1, Hq=1, Hkv=1, L=64, d=16, seed=29)
    ref, _ = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    _, _, pm, pl, po = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), None, p.scale, 4)
    m = pm[0, 0].max()
    w = np.exp(pm[0, 0] - m) * pl[0, 0]
    good = (w[:, None] * po[0, 0]).sum(0) / w.sum()
    bad = (w[:, None] * (po[0, 0] * pl[0, 0][:, None])).sum(0) / w.sum()
    np.testing.assert_allclose(good, ref[0, 0], atol=1e-12)
    assert np.abs(bad - ref[0, 0]).max() > 1e-3


def test_page_demo_shape_split_invariance(oracle):
    # the tutorial's numpy demo shape: seed 42, d=64, n=16384, 4 blocks, scale 1/sqrt(d)
    with open(os.path.join(GOLDEN, "pages_fixtures.json")) as f:
        demo = json.load(f)["flash_decoding_demo"]
    n, d, S = demo["n"], demo["d"], demo["num_blocks"]
    p = W.random_problem(1, 1, 1, n, d, seed=demo["seed"], scale=1.0 / math.sqrt(d))
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    out, lse, *_ = oracle.decode_split(bits(p.q), bits(p.k), bits(p.v), None, p.scale, S)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lref, atol=1e-12)


# ------------------------------------------------------------------- paging

def test_token_permutation_invariance(oracle):
    p = small(B=1, Hq=2, Hkv=1, L=33, d=16, seed=31)
    perm = torch.randperm(33, generator=torch.Generator().manual_seed(1))
    out1, l1 = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    out2, l2 = oracle.decode_dense(bits(p.q), bits(p.k[:, :, perm]), bits(p.v[:, :, perm]), None, p.scale)
    np.testing.assert_allclose(out1, out2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("identity", [True, False])
def test_paged_equals_contiguous(oracle, identity):
    p = small(B=3, Hq=4, Hkv=2, L=200, d=16, seed=37, seq_lens=[200, 64, 1])
    pp = W.to_paged(p, identity=identity, page_size=64)
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens, p.scale)
    out, lse = oracle.decode_paged(bits(pp.q), bits(pp.k_pages), bits(pp.v_pages), pp.page_table,
                                   pp.num_pages, pp.seq_lens, pp.scale)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, lref)


def test_paged_rejects_bad_page_id(oracle):
    p = small(B=1, Hq=1, Hkv=1, L=100, d=16, seed=41)
    pp = W.to_paged(p, page_size=64)
    table = pp.page_table.clone()
    table[0, 1] = pp.num_pages
    with pytest.raises(ValueError):
        oracle.decode_paged(bits(pp.q), bits(pp.k_pages), bits(pp.v_pages), table, pp.num_pages,
                            pp.seq_lens, pp.scale)
