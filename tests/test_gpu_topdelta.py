"""GPU parity of the key encoder and the fused top-delta decode.

Encoder: codes, fp16 min/scale, int8 residuals and fp16 residual scales must
equal the oracle's bit for bit (both evaluate the same binary32 definition).

Top-delta: the GPU decodes from the ORACLE's encoding of the keys (so the
oracle never sees a value the CUDA path produced); the candidate set per
(sequence, query head) must equal the oracle's exactly, except at tokens whose
2-bit score lies within 1e-4 of the threshold m^ - delta (ties: both choices
are valid, they are counted and reported).  Outputs: bf16 within
1e-2 * (1 + |ref|), fp32 within 1e-4 * (1 + |ref|), LSE within 1e-3; a row
whose set differs at a tie is held to that bound plus the weight the
differing tokens carry.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from parity import BF16_TOL, F32_TOL, LSE_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIE = 1e-4


def to_dev(enc):
    codes, ms, res, rs = enc
    return (torch.from_numpy(codes).to(DEV), torch.from_numpy(ms.view(np.float16)).to(DEV),
            torch.from_numpy(res).to(DEV), torch.from_numpy(rs.view(np.float16)).to(DEV))


def mask_bits(mask_words, L):
    w = np.asarray(mask_words, np.uint32)
    bitsarr = ((w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)
    return bitsarr.reshape(*w.shape[:-1], -1)[..., :L]


# ------------------------------------------------------------------ encoder

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("std", [1.0, 1e-3, 40.0])
def test_encoder_bit_exact(fd, oracle, d, std):
    lens = [333, 0, 1000]
    p = W.random_problem(3, 4, 4, 1000, d, seed=int(std * 10) + d, device=DEV, std=std, seq_lens=lens)
    k = p.k.clone()
    # special groups: constant, grid-aligned, ties at half steps, signed zero
    k[0, 0, 0, :32] = 0.75
    k[0, 0, 1, :32] = torch.tensor([-1.0, 0.0, 1.0, 2.0] * 8)
    k[0, 0, 2, :32] = torch.tensor([0.0, 3.0, 0.5, 1.5, 2.5] + [0.0] * 27)
    k[0, 0, 3, :32] = -0.0
    k[0, 0, 4, :32] = torch.tensor([-0.0, 0.0] * 16)
    ref = oracle.quantize_keys(bits(k), p.seq_lens.cpu())
    got = fd.fd_quantize_keys(k, p.seq_lens)
    torch.cuda.synchronize()
    for b, L in enumerate(lens):
        for name, r, g in zip(("codes", "mn_scale", "res", "res_scale"), ref, got):
            gv = g[b, :, :L].cpu().numpy()
            if gv.dtype == np.float16:
                gv = gv.view(np.uint16)
            np.testing.assert_array_equal(gv, r[b, :, :L], err_msg=f"{name} b={b}")


def test_encoder_full_ffd_sample(fd, oracle):
    """Full FFD workload keys: the GPU encoding of two KV heads equals the oracle's."""
    p = W.ffd(seed=0, device=DEV)
    enc = fd.fd_quantize_keys(p.k, p.seq_lens)
    torch.cuda.synchronize()
    for h in (0, 7):
        ref = oracle.quantize_keys(bits(p.k[:, h:h + 1]))
        for r, g in zip(ref, enc):
            gv = g[:, h:h + 1].cpu().numpy()
            if gv.dtype == np.float16:
                gv = gv.view(np.uint16)
            np.testing.assert_array_equal(gv, r)


# -------------------------------------------------------------- top-delta

def run_both(fd, oracle, p, delta, n_sink=4, window=64, num_splits=0, out_dtype="bf16", group_union=False):
    sl = p.seq_lens
    enc = oracle.quantize_keys(bits(p.k), sl.cpu())
    ref_fn = oracle.decode_topdelta_group_union if group_union else oracle.decode_topdelta
    ref = ref_fn(bits(p.q), *enc, bits(p.v), sl.cpu(), p.scale, delta, n_sink, window, want_scores=True)
    c, ms, r, rs = to_dev(enc)
    out, lse, mask, cnt = fd.fd_decode_topdelta(p.q, c, ms, r, rs, p.v, sl, p.scale, delta, n_sink, window,
                                                num_splits=num_splits, out_dtype=out_dtype, want_selection=True,
                                                group_union=group_union)
    torch.cuda.synchronize()
    return enc, ref, out, lse, mask.cpu().numpy().view(np.uint32), cnt.cpu().numpy()


def check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, delta, tol, group_union=False):
    L_max = p.L_max
    lens = p.seq_lens.cpu().numpy()
    got_sel = mask_bits(mask, L_max)
    ref_sel = mask_bits(ref["sel_mask"], L_max)
    st = ref["s_tilde"]
    thr = ref["m_hat"][..., None] - delta
    ties = 0
    kt = None
    G = p.Hq // p.Hkv
    out_np = out.float().cpu().numpy().astype(np.float64)
    lse_np = lse.cpu().numpy().astype(np.float64)
    for b in range(p.B):
        L = int(lens[b])
        for hq in range(p.Hq):
            diff = np.nonzero(got_sel[b, hq, :L] != ref_sel[b, hq, :L])[0]
            if diff.size:
                # a token may differ only at a tie: of this head, or (shared sets) of any head of its group
                heads = range((hq // G) * G, (hq // G + 1) * G) if group_union else (hq,)
                near = np.zeros(diff.size, bool)
                for g in heads:
                    near |= np.abs(st[b, g, diff] - thr[b, g, 0]) <= TIE
                assert near.all(), f"selection differs away from the threshold at b={b} hq={hq} j={diff[~near]}"
                ties += diff.size
            assert cnt[b, hq] == int(got_sel[b, hq, :L].sum())
            assert not got_sel[b, hq, L:].any()
            ref_o = ref["out"][b, hq]
            slack = 0.0
            if diff.size:
                # weight of the tie tokens whose membership differs bounds the output change
                if kt is None:
                    kt = oracle.dequantize_keys(*enc, seq_lens=p.seq_lens.cpu())
                s = p.scale * (kt[b, hq // G, diff] @ p.q[b, hq].double().cpu().numpy())
                wsum = float(np.exp(s - ref["lse"][b, hq]).sum())
                vmax = float(p.v[b, hq // G, :L].abs().max())
                slack = 2.0 * wsum * vmax / max(1e-30, 1.0 - wsum)
                assert abs(lse_np[b, hq] - ref["lse"][b, hq]) <= LSE_TOL + 2.0 * wsum
            else:
                if np.isneginf(ref["lse"][b, hq]):
                    assert np.isneginf(lse_np[b, hq])
                else:
                    assert abs(lse_np[b, hq] - ref["lse"][b, hq]) <= LSE_TOL
            err = np.abs(out_np[b, hq] - ref_o)
            assert np.all(err <= tol * (1 + np.abs(ref_o)) + slack), (b, hq, err.max(), slack)
    return ties


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("delta", [5.0, 7.0])
def test_topdelta_parity_small(fd, oracle, d, G, delta):
    Hkv = 2
    p = W.ffd(seed=G * 3 + d, B=2, L=2500, Hq=Hkv * G, Hkv=Hkv, d=d)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.seq_lens.to(DEV), p.scale, p.L_max)
    for ns in (0, 1, 3):
        enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, delta, num_splits=ns)
        check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, delta, BF16_TOL)


def test_topdelta_ragged_and_empty(fd, oracle):
    lens = [0, 5, 64, 68, 130, 1000, 2048]
    p = W.random_problem(len(lens), 8, 2, 2048, 128, seed=31, device=DEV, seq_lens=lens)
    for delta in (0.0, 2.0, math.inf):
        enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, delta, out_dtype="f32")
        check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, delta, F32_TOL)
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_topdelta_infinite_delta_is_dense_over_dequantized_keys(fd, oracle):
    p = W.ffd(seed=5, B=2, L=3000, Hq=8, Hkv=2, d=128)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.seq_lens.to(DEV), p.scale, p.L_max)
    enc = oracle.quantize_keys(bits(p.k))
    c, ms, r, rs = to_dev(enc)
    out, lse, _, cnt = fd.fd_decode_topdelta(p.q, c, ms, r, rs, p.v, None, p.scale, math.inf,
                                             out_dtype="f32", want_selection=True)
    kt = oracle.dequantize_keys(*enc)
    ref, lref = oracle.decode_dense_f64(p.q.double().cpu().numpy(), kt, p.v.double().cpu().numpy(), None, p.scale)
    assert_out_close(out, ref, F32_TOL)
    assert_lse_close(lse, lref)
    assert torch.all(cnt == 3000)


def test_topdelta_deterministic_and_split_invariant(fd, oracle):
    # the same inputs and chunk count give the same bits (selection bits and counts are
    # order-free atomics, the arithmetic order is fixed); other chunk counts change the
    # output only by fp32 rounding and leave the selection untouched
    p = W.ffd(seed=9, B=2, L=6000, Hq=8, Hkv=2, d=128)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.seq_lens.to(DEV), p.scale, p.L_max)
    c, ms, r, rs = to_dev(oracle.quantize_keys(bits(p.k)))
    runs = {}
    for ns in (1, 3, 7, 0, 3):
        runs.setdefault(ns, []).append(
            fd.fd_decode_topdelta(p.q, c, ms, r, rs, p.v, None, p.scale, 5.0, num_splits=ns, out_dtype="f32",
                                  want_selection=True))
    a, b = runs[3]
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    out0, lse0, mask0, cnt0 = runs[1][0]
    for ns in (3, 7, 0):
        out, lse, mask, cnt = runs[ns][0]
        assert torch.equal(mask, mask0) and torch.equal(cnt, cnt0)
        assert (out - out0).abs().max().item() < 1e-5
        assert (lse - lse0).abs().max().item() < 1e-5


def crafted_dev(mn_values, d=64):
    """2-bit body constant mn_t on every channel (s16 = 0): with q = 1/d and
    scale 1 the 2-bit score is exactly mn_t."""
    L = len(mn_values)
    codes = torch.zeros((1, 1, L, d // 4), dtype=torch.uint8)
    ms = torch.zeros((1, 1, L, d // 32, 2), dtype=torch.float16)
    ms[..., 0] = torch.tensor(mn_values, dtype=torch.float16)[None, None, :, None]
    res = torch.zeros((1, 1, L, d), dtype=torch.int8)
    rs = torch.zeros((1, 1, L, d // 32), dtype=torch.float16)
    q = torch.full((1, 1, d), 1.0 / d).to(torch.bfloat16)
    v = torch.randn((1, 1, L, d), generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    return [t.to(DEV) for t in (q, codes, ms, res, rs, v)]


def test_topdelta_pseudo_max_and_inclusive_threshold(fd):
    # anchors of L=200 with 4 sinks and a 64-token window: {0..3} U {136..199}
    mn = np.full(200, -8.0)
    mn[2], mn[136], mn[150] = 1.0, 1.5, 1.25
    mn[100], mn[4], mn[135] = 4.0, 3.0, 3.0
    mn[50], mn[51] = -3.5, -3.50390625
    q, c, ms, r, rs, v = crafted_dev(list(mn))
    out, lse, mask, cnt = fd.fd_decode_topdelta(q, c, ms, r, rs, v, None, 1.0, 5.0, 4, 64, out_dtype="f32",
                                                want_selection=True)
    sel = np.nonzero(mask_bits(mask.cpu().numpy().view(np.uint32), 200)[0, 0])[0].tolist()
    assert sel == [2, 4, 50, 100, 135, 136, 150]
    s = mn[sel]
    w = np.exp(s - s.max())
    w /= w.sum()
    np.testing.assert_allclose(out[0, 0].cpu().numpy(), w @ v[0, 0, sel].double().cpu().numpy(), atol=1e-5)
    assert abs(float(lse[0, 0]) - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-5


def test_topdelta_full_ffd_sampled(fd, oracle):
    """The full FFD workload (B=4, Hq=32, Hkv=8, d=128, L=131072) at delta 5 and 7
    in the benchmark's launch configuration; oracle on two KV heads."""
    p = W.ffd(seed=0, device=DEV)
    enc_gpu = fd.fd_quantize_keys(p.k, p.seq_lens)
    G = p.Hq // p.Hkv
    for delta in (5.0, 7.0):
        out, lse, mask, cnt = fd.fd_decode_topdelta(p.q, *enc_gpu, p.v, p.seq_lens, p.scale, delta,
                                                    want_selection=True)
        torch.cuda.synchronize()
        mask = mask.cpu().numpy().view(np.uint32)
        cnt = cnt.cpu().numpy()
        ties = 0
        for h in (0, 7):
            sub = W.Problem("ffd_sub", p.q[:, h * G:(h + 1) * G].contiguous(), p.k[:, h:h + 1].contiguous(),
                            p.v[:, h:h + 1].contiguous(), p.seq_lens, p.scale, p.L_max)
            enc = oracle.quantize_keys(bits(sub.k))
            # the GPU decoded from its own encoding: identical to the oracle's, bit for bit
            for rr, g in zip(enc, enc_gpu):
                gv = g[:, h:h + 1].cpu().numpy()
                np.testing.assert_array_equal(gv.view(np.uint16) if gv.dtype == np.float16 else gv, rr)
            ref = oracle.decode_topdelta(bits(sub.q), *enc, bits(sub.v), None, p.scale, delta, 4, 64,
                                         want_scores=True)
            ties += check_topdelta(oracle, sub, enc, ref, out[:, h * G:(h + 1) * G], lse[:, h * G:(h + 1) * G],
                                   mask[:, h * G:(h + 1) * G], cnt[:, h * G:(h + 1) * G], delta, BF16_TOL)
        print(f"delta={delta}: tie tokens with differing membership: {ties}")


def test_topdelta_million_tokens_sampled(fd, oracle):
    """The 1M-token GQA cache (B=1, Hq=32, Hkv=8, d=128, sinks +3 q^) at delta 5: the planner's many
    chunks per (sequence, head), the anchor window a million tokens past the sinks; oracle on two KV
    heads."""
    p = W.million(seed=0, device=DEV)
    enc_gpu = fd.fd_quantize_keys(p.k, None)
    G = p.Hq // p.Hkv
    delta = 5.0
    out, lse, mask, cnt = fd.fd_decode_topdelta(p.q, *enc_gpu, p.v, None, p.scale, delta, want_selection=True)
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    mask = mask.cpu().numpy().view(np.uint32)
    cnt = cnt.cpu().numpy()
    for h in (0, 5):
        sub = W.Problem("million_sub", p.q[:, h * G:(h + 1) * G].contiguous(), p.k[:, h:h + 1].contiguous(),
                        p.v[:, h:h + 1].contiguous(), p.seq_lens, p.scale, p.L_max)
        enc = oracle.quantize_keys(bits(sub.k))
        for rr, g in zip(enc, enc_gpu):
            gv = g[:, h:h + 1].cpu().numpy()
            np.testing.assert_array_equal(gv.view(np.uint16) if gv.dtype == np.float16 else gv, rr)
        ref = oracle.decode_topdelta(bits(sub.q), *enc, bits(sub.v), None, p.scale, delta, 4, 64, want_scores=True)
        check_topdelta(oracle, sub, enc, ref, out[:, h * G:(h + 1) * G], lse[:, h * G:(h + 1) * G],
                       mask[:, h * G:(h + 1) * G], cnt[:, h * G:(h + 1) * G], delta, BF16_TOL)


# ------------------------------------------------- anchor settings, shared sets

@pytest.mark.parametrize("n_sink", [0, 1, 16, 64])
@pytest.mark.parametrize("window", [0, 16, 256, 1024])
def test_topdelta_anchor_settings(fd, oracle, n_sink, window):
    """The sink counts and window lengths the anchor sweep times, against the
    oracle: they move the anchor pass's tile walk (sink tiles, the jump to the
    window, windows longer than the sequence, no anchors at all: m^ = -inf,
    everything selected)."""
    p = W.ffd(seed=17, B=4, L=2500, Hq=8, Hkv=2, d=128)
    lens = torch.tensor([2500, 700, 5, 0], dtype=torch.int32)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), lens.to(DEV), p.scale, p.L_max)
    enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, 5.0, n_sink, window)
    check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, 5.0, BF16_TOL)
    if n_sink == 0 and window == 0:
        assert np.array_equal(cnt, np.repeat(lens.numpy()[:, None], p.Hq, axis=1))


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("delta", [2.0, 5.0])
def test_topdelta_group_union_parity(fd, oracle, G, delta):
    Hkv = 2
    p = W.ffd(seed=23 + G, B=2, L=3000, Hq=Hkv * G, Hkv=Hkv, d=128)
    lens = torch.tensor([3000, 1234], dtype=torch.int32)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), lens.to(DEV), p.scale, p.L_max)
    for ns, dt, tol in ((0, "bf16", BF16_TOL), (3, "f32", F32_TOL)):
        enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, delta, num_splits=ns, out_dtype=dt,
                                                 group_union=True)
        check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, delta, tol, group_union=True)
        # one set per group
        m = mask.reshape(p.B, Hkv, G, -1)
        assert np.all(m == m[:, :, :1])


def test_topdelta_sparse_cache_skips_tiles(fd, oracle):
    """A sparse cache (anchors and 0.2% planted tokens far above
    the rest): few 64-token tiles hold a candidate, so the residual and V of
    most tiles are never read; sets and outputs still match the oracle."""
    p = W.ffd(seed=29, B=2, L=8192, Hq=8, Hkv=2, d=128, anchor_boost=20.0, plant_mean=20.0, plant_frac=0.002)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.seq_lens.to(DEV), p.scale, p.L_max)
    for group_union in (False, True):
        enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, 5.0, group_union=group_union)
        check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, 5.0, BF16_TOL, group_union=group_union)
        sel = mask_bits(mask, p.L_max).reshape(p.B, p.Hkv, p.Hq // p.Hkv, -1).any(axis=2)
        tiles = sel.reshape(p.B, p.Hkv, -1, 64).any(axis=-1)
        assert tiles.mean() < 0.25, tiles.mean()
