"""GPU parity of the fp4 (e2m1, power-of-two block scales) KV cache path
against the CPU oracle.

The encoder must reproduce the oracle's codes and scale bytes bit for bit.
The decode is fed the oracle's own codes and compared with the oracle's
binary64 attention over the decoded rows: bf16 outputs within
1e-2 * (1 + |ref|), LSE within 1e-3, fp32 outputs within the bound of the
kernel's arithmetic (its only rounding above fp32 level is the fp16 operand
P * 2^e / s_ref, relative 2^-11): 2^-11 * max|v~| + 1e-4 * (1 + |ref|).
"""
import numpy as np
import pytest
import torch

import workloads as W
from parity import BF16_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def oracle_codes(oracle, x, seq_lens=None):
    c, s = oracle.quantize_kv_fp4(bits(x), None if seq_lens is None else seq_lens.cpu())
    return torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV)


def oracle_vcodes(oracle, x, seq_lens=None):
    c, s = oracle.quantize_v_fp4(bits(x), None if seq_lens is None else seq_lens.cpu())
    return torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV)


def fp4_problem(oracle, p):
    return oracle_codes(oracle, p.k) + oracle_vcodes(oracle, p.v)


def poison_value_tail(vc, b, L):
    """Codes 0xF (-6) for every value token at or past L of sequence b."""
    vc[b, :, (L + 1) // 2:] = 0xFF
    if L % 2:
        vc[b, :, L // 2] |= 0xF0


def oracle_fp4(oracle, p, kc, ks, vc, vs, seq_lens=True):
    return oracle.decode_dense_fp4(bits(p.q), kc.cpu().numpy(), ks.cpu().numpy(), vc.cpu().numpy(),
                                   vs.cpu().numpy(), p.seq_lens.cpu() if seq_lens else None, p.scale)


def f32_bound_check(out, ref, vc, vs, oracle):
    vmax = np.abs(oracle.dequantize_v_fp4(vc.cpu().numpy(), vs.cpu().numpy())).max()
    g = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    assert np.all(err <= 2.0**-11 * vmax + 1e-4 * (1 + np.abs(ref))), err.max()


# ------------------------------------------------------------------ encoder

@pytest.mark.parametrize("d", [64, 128])
def test_encoder_bit_exact(fd, oracle, d):
    g = torch.Generator().manual_seed(d + 1)
    B, H, L = 3, 2, 300
    mag = torch.exp2(torch.empty(B, H, L, 1).uniform_(-40, 40, generator=g))
    x = (torch.randn(B, H, L, d, generator=g) * mag).to(torch.bfloat16)
    x[0, 0, 5] = 0.0                                   # all-zero row
    x[0, 0, 6, ::2] = -0.0                             # signed zeros
    x[0, 0, 7, :32] = -1e-3                            # values far below the block maximum
    x[0, 0, 7, 0] = 6.0
    x[1, 1, 7, :8] = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])  # e = 0, ties
    x[1, 1, 7, 8:16] = -x[1, 1, 7, :8]
    x[2, 0, 9, 0] = 1e-38                              # a subnormal block maximum
    x[2, 0, 9, 1:] = 0
    x = x.to(DEV)
    sl = torch.tensor([300, 123, 0], dtype=torch.int32, device=DEV)
    codes = torch.full((B, H, L, d // 2), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((B, H, L, d // 32), 0xCD, dtype=torch.uint8, device=DEV)
    fd.fd_quantize_kv_fp4(x, sl, codes=codes, scales=scales)
    rc, rs = oracle.quantize_kv_fp4(bits(x), sl.cpu())
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    for b, L_b in enumerate(sl.tolist()):
        np.testing.assert_array_equal(c[b, :, :L_b], rc[b, :, :L_b])
        np.testing.assert_array_equal(s[b, :, :L_b], rs[b, :, :L_b])
        assert np.all(c[b, :, L_b:] == 0xAB) and np.all(s[b, :, L_b:] == 0xCD)  # untouched
    assert fd.fd_device_status(clear=True) == fd.FD_OK


@pytest.mark.parametrize("d", [64, 128])
def test_value_encoder_bit_exact(fd, oracle, d):
    g = torch.Generator().manual_seed(d + 7)
    B, H, L = 3, 2, 301                                # odd L_max: the last pair of a head is half empty
    mag = torch.exp2(torch.empty(B, H, L, 1).uniform_(-40, 40, generator=g))
    x = (torch.randn(B, H, L, d, generator=g) * mag).to(torch.bfloat16)
    x[0, 0, 4] = 0.0
    x[0, 0, 5, ::2] = -0.0
    x[1, 1, 6, :8] = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    x = x.to(DEV)
    sl = torch.tensor([301, 124, 0], dtype=torch.int32, device=DEV)
    codes = torch.full((B, H, (L + 1) // 2, d), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((B, H, L, d // 32), 0xCD, dtype=torch.uint8, device=DEV)
    fd.fd_quantize_v_fp4(x, sl, codes=codes, scales=scales)
    rc, rs = oracle.quantize_v_fp4(bits(x), sl.cpu())
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    for b, L_b in enumerate(sl.tolist()):
        P_b = (L_b + 1) // 2
        np.testing.assert_array_equal(c[b, :, :P_b], rc[b, :, :P_b])
        np.testing.assert_array_equal(s[b, :, :L_b], rs[b, :, :L_b])
        assert np.all(c[b, :, P_b:] == 0xAB) and np.all(s[b, :, L_b:] == 0xCD)  # untouched
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_encoder_full_size_sampled(fd, oracle):
    p = W.mha32k(seed=0, device=DEV)
    codes, scales = fd.fd_quantize_kv_fp4(p.k)
    vcodes, vscales = fd.fd_quantize_v_fp4(p.v)
    for h in (0, 19):
        rc, rs = oracle.quantize_kv_fp4(bits(p.k[:, h:h + 1]))
        np.testing.assert_array_equal(codes[:, h:h + 1].cpu().numpy(), rc)
        np.testing.assert_array_equal(scales[:, h:h + 1].cpu().numpy(), rs)
        rc, rs = oracle.quantize_v_fp4(bits(p.v[:, h:h + 1]))
        np.testing.assert_array_equal(vcodes[:, h:h + 1].cpu().numpy(), rc)
        np.testing.assert_array_equal(vscales[:, h:h + 1].cpu().numpy(), rs)


# ------------------------------------------------------------------ decode

SHAPES = [
    # B, Hq, Hkv, L, d
    (1, 1, 1, 1, 64),
    (1, 1, 1, 65, 128),
    (2, 4, 4, 1000, 128),
    (3, 8, 2, 777, 128),
    (2, 6, 2, 301, 64),      # group 3, L_max not a multiple of 4
    (2, 8, 1, 513, 128),     # group 8
    (1, 16, 2, 2049, 64),    # group 8, d 64
    (2, 12, 4, 4099, 128),   # group 3
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_Hq%d_Hkv%d_L%d_d%d" % s)
@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_fp4_decode_parity_small(fd, oracle, shape, num_splits):
    B, Hq, Hkv, L, d = shape
    p = W.random_problem(B, Hq, Hkv, L, d, seed=sum(shape) % 991, device=DEV)
    kc, ks, vc, vs = fp4_problem(oracle, p)
    ref, lref = oracle_fp4(oracle, p, kc, ks, vc, vs, seq_lens=False)
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale, num_splits=num_splits)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    out32, lse32 = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale, num_splits=num_splits,
                                          out_dtype="f32")
    f32_bound_check(out32, ref, vc, vs, oracle)
    assert_lse_close(lse32, lref, 1e-4)


@pytest.mark.parametrize("d", [64, 128])
def test_fp4_ragged_empty_and_poisoned_tails(fd, oracle, d):
    lens = [0, 1, 63, 64, 65, 1000, 2047, 2048]
    p = W.random_problem(len(lens), 8, 2, 2048, d, seed=22, device=DEV, seq_lens=lens)
    kc, ks, vc, vs = fp4_problem(oracle, p)
    ref, lref = oracle_fp4(oracle, p, kc, ks, vc, vs)
    for b, L in enumerate(lens):  # -6 codes and infinite scales (byte 255) past each end
        kc[b, :, L:] = 0xFF
        poison_value_tail(vc, b, L)
        ks[b, :, L:] = 0xFF
        vs[b, :, L:] = 0xFF
    for ns in (0, 1, 5):
        out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, p.seq_lens, p.scale, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)
        assert torch.all(out[0] == 0)


def test_fp4_split_invariance_and_determinism(fd, oracle):
    p = W.random_problem(2, 8, 2, 5000, 128, seed=6, device=DEV)
    kc, ks, vc, vs = fp4_problem(oracle, p)
    ref, lref = oracle_fp4(oracle, p, kc, ks, vc, vs, seq_lens=False)
    for ns in (1, 2, 3, 8, 40, 79, 0):
        out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale, num_splits=ns, out_dtype="f32")
        f32_bound_check(out, ref, vc, vs, oracle)
        assert_lse_close(lse, lref, 1e-4)
    a, la = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale)
    b, lb = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_fp4_extreme_scales(fd, oracle):
    # block scales spread over 2^-60 .. 2^60 (per row and per block) and a large query
    p = W.random_problem(1, 4, 1, 900, 128, seed=32, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(4)
    kmag = torch.exp2(torch.empty(1, 1, 900, 4, 1, device=DEV).uniform_(-20, 20, generator=g))
    vmag = torch.exp2(torch.empty(1, 1, 900, 4, 1, device=DEV).uniform_(-60, 60, generator=g))
    p.k = (p.k.float().view(1, 1, 900, 4, 32) * kmag * 1e-3).view(1, 1, 900, 128).to(torch.bfloat16)
    p.v = (p.v.float().view(1, 1, 900, 4, 32) * vmag).view(1, 1, 900, 128).to(torch.bfloat16)
    p.q = (p.q.float() * 3e4).to(torch.bfloat16)
    kc, ks, vc, vs = fp4_problem(oracle, p)
    ref, lref = oracle_fp4(oracle, p, kc, ks, vc, vs, seq_lens=False)
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale, out_dtype="f32")
    f32_bound_check(out, ref, vc, vs, oracle)
    assert np.allclose(lse.cpu().numpy(), lref, rtol=1e-5, atol=1e-3)


def test_fp4_gpu_encoder_then_decode(fd, oracle):
    p = W.random_problem(2, 8, 2, 3000, 128, seed=42, device=DEV, seq_lens=[3000, 1234])
    kc, ks = fd.fd_quantize_kv_fp4(p.k, p.seq_lens)
    vc, vs = fd.fd_quantize_v_fp4(p.v, p.seq_lens)
    ref, lref = oracle_fp4(oracle, p, *fp4_problem(oracle, p))
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, p.seq_lens, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)


# ------------------------------------------------------------------- paged

def paged_codes(oracle, pp, lens):
    kc, ks = oracle_codes(oracle, pp.k_pages)
    vc, vs = oracle_vcodes(oracle, pp.v_pages)  # pages [P, Hkv, 64, d] -> pair pages [P, Hkv, 32, d]
    for b, L in enumerate(lens):
        if L % 64:
            pid = int(pp.page_table[b, (L - 1) // 64])
            for t in (kc, ks, vs):
                t[pid, :, L % 64:] = 0xFF
            poison_value_tail(vc, pid, L % 64)
    return kc, ks, vc, vs


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_fp4_paged_parity(fd, oracle, G, d):
    lens = [1, 64, 65, 700, 3000, 0]
    Hkv = 2
    p = W.random_problem(len(lens), Hkv * G, Hkv, 3000, d, seed=G + d + 1, device=DEV, seq_lens=lens)
    pp = W.to_paged(p, seed=3, poison_tail=False)
    kc, ks, vc, vs = paged_codes(oracle, pp, lens)
    ref, lref = oracle_fp4(oracle, p, *fp4_problem(oracle, p))
    for ns in (0, 1, 4):
        out, lse = fd.fd_decode_paged_fp4(pp.q, kc, ks, vc, vs, pp.page_table, pp.num_pages, pp.seq_lens,
                                          pp.scale, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_fp4_paged_bad_page_is_reported(fd, oracle):
    # a page id past the pool is reported and not read; the other sequence is unaffected
    lens = [300, 200]
    p = W.random_problem(2, 8, 2, 300, 128, seed=9, device=DEV, seq_lens=lens)
    pp = W.to_paged(p, seed=4, poison_tail=False)
    kc, ks, vc, vs = paged_codes(oracle, pp, lens)
    ref, lref = oracle_fp4(oracle, p, *fp4_problem(oracle, p))
    table = pp.page_table.clone()
    table[1, 2] = pp.num_pages + 5
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    out, lse = fd.fd_decode_paged_fp4(pp.q, kc, ks, vc, vs, table, pp.num_pages, pp.seq_lens, pp.scale)
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_BAD_PAGE_TABLE
    assert torch.isfinite(out.float()).all()
    assert_out_close(out[:1], ref[:1], BF16_TOL)
    assert_lse_close(lse[:1], lref[:1])


# --------------------------------------------------------- full workloads

def test_fp4_full_mha32k_sampled(fd, oracle):
    p = W.mha32k(seed=0, device=DEV)
    kc, ks = fd.fd_quantize_kv_fp4(p.k)
    vc, vs = fd.fd_quantize_v_fp4(p.v)
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale)
    for h in (0, 13, 31):
        sl = slice(h, h + 1)
        ref, lref = oracle.decode_dense_fp4(bits(p.q[:, sl]), kc[:, sl].cpu().numpy(), ks[:, sl].cpu().numpy(),
                                            vc[:, sl].cpu().numpy(), vs[:, sl].cpu().numpy(), None, p.scale)
        assert_out_close(out[:, sl], ref, BF16_TOL, what=f"head {h}")
        assert_lse_close(lse[:, sl], lref)


def test_fp4_full_gqa_sampled(fd, oracle):
    p = W.ffd(seed=0, device=DEV)
    kc, ks = fd.fd_quantize_kv_fp4(p.k)
    vc, vs = fd.fd_quantize_v_fp4(p.v)
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, None, p.scale)
    G = p.Hq // p.Hkv
    for h in (0, 5):
        ks_ = slice(h, h + 1)
        qs = slice(h * G, (h + 1) * G)
        ref, lref = oracle.decode_dense_fp4(bits(p.q[:, qs]), kc[:, ks_].cpu().numpy(), ks[:, ks_].cpu().numpy(),
                                            vc[:, ks_].cpu().numpy(), vs[:, ks_].cpu().numpy(), None, p.scale)
        assert_out_close(out[:, qs], ref, BF16_TOL, what=f"kv head {h}")
        assert_lse_close(lse[:, qs], lref)


def test_fp4_many_short_ragged_sequences(fd, oracle):
    B = 3000
    g = torch.Generator().manual_seed(14)
    lens = torch.randint(0, 201, (B,), generator=g).tolist()
    p = W.random_problem(B, 8, 2, 200, 128, seed=14, device=DEV, seq_lens=lens)
    kc, ks = fd.fd_quantize_kv_fp4(p.k, p.seq_lens)
    vc, vs = fd.fd_quantize_v_fp4(p.v, p.seq_lens)
    ref, lref = oracle_fp4(oracle, p, kc, ks, vc, vs)
    out, lse = fd.fd_decode_dense_fp4(p.q, kc, ks, vc, vs, p.seq_lens, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
