"""GPU parity of the dense and paged split-KV decode against the CPU oracle.

Every case runs the C-ABI library through its binding on seeded inputs and
compares element by element with the fp64 oracle: bf16 outputs within
1e-2 * (1 + |ref|), fp32 outputs within 1e-4 * (1 + |ref|), LSE within 1e-3.
Small shapes span several 64-token tiles, ragged tails, empty sequences,
every group size up to 8 and explicit and planned chunk counts; the full
workload sizes run in the planner's launch configuration (the one the
benchmark times) with the oracle on a sample of heads.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from parity import BF16_TOL, F32_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def oracle_dense(oracle, p):
    return oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)


def run_dense(fd, p, out_dtype="bf16", num_splits=None, seq_lens=True):
    return fd.fd_decode_dense(p.q, p.k, p.v, p.seq_lens if seq_lens else None, p.scale,
                              num_splits=p.num_splits if num_splits is None else num_splits,
                              out_dtype=out_dtype)


SHAPES = [
    # B, Hq, Hkv, L, d
    (1, 1, 1, 1, 64),
    (1, 1, 1, 65, 128),
    (2, 4, 4, 1000, 128),
    (3, 8, 2, 777, 128),
    (2, 6, 2, 300, 64),      # group 3 (padded to 4)
    (2, 8, 1, 513, 128),     # group 8
    (1, 16, 2, 2049, 64),    # group 8, d 64
    (2, 12, 4, 4100, 128),   # group 3
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_Hq%d_Hkv%d_L%d_d%d" % s)
@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_dense_parity_small(fd, oracle, shape, num_splits):
    B, Hq, Hkv, L, d = shape
    p = W.random_problem(B, Hq, Hkv, L, d, seed=hash(shape) % 1000, device=DEV)
    ref, lref = oracle_dense(oracle, p)
    out, lse = run_dense(fd, p, num_splits=num_splits, seq_lens=False)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("d", [64, 128])
def test_dense_ragged_lengths_and_empty(fd, oracle, d):
    lens = [0, 1, 63, 64, 65, 1000, 2047, 2048]
    p = W.random_problem(len(lens), 8, 2, 2048, d, seed=11, device=DEV, seq_lens=lens)
    # poison everything past each sequence's end: it must never be read
    for b, L in enumerate(lens):
        p.k[b, :, L:] = float("nan")
        p.v[b, :, L:] = float("nan")
    ref, lref = oracle_dense(oracle, p)
    for ns in (0, 1, 5):
        out, lse = run_dense(fd, p, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)
        assert torch.all(out[0] == 0)


def test_tiny_workload_fp32(fd, oracle):
    # B=1, Hq=Hkv=1, d=64, L=1024, scale 1/8, 4 chunks, fp32 output + LSE
    p = W.tiny(seed=0, device=DEV)
    ref, lref = oracle_dense(oracle, p)
    out, lse = run_dense(fd, p, out_dtype="f32")
    assert fd.fd_num_splits(1, 1, 1, 1024, 64, 4) == 4
    assert_out_close(out, ref, F32_TOL)
    assert_lse_close(lse, lref, 1e-5)


def test_split_count_invariance(fd, oracle):
    p = W.random_problem(2, 8, 2, 5000, 128, seed=5, device=DEV)
    ref, lref = oracle_dense(oracle, p)
    outs = []
    for ns in (1, 2, 3, 8, 40, 79, 0):
        out, lse = run_dense(fd, p, out_dtype="f32", num_splits=ns, seq_lens=False)
        assert_out_close(out, ref, F32_TOL)
        assert_lse_close(lse, lref, 1e-5)
        outs.append(out)
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 1e-4


@pytest.mark.parametrize("d", [64, 128])
def test_merge_of_more_chunks_than_threads(fd, oracle, d):
    # the merge kernel runs d threads per row and takes the chunk weights d at
    # a time: 157 chunks of 128 tokens (and fewer for the shorter sequence)
    # cross that block boundary at both head sizes
    p = W.random_problem(2, 4, 2, 20000, d, seed=12 + d, device=DEV, seq_lens=[20000, 9000])
    ref, lref = oracle_dense(oracle, p)
    out, lse = run_dense(fd, p, out_dtype="f32", num_splits=300)
    assert_out_close(out, ref, F32_TOL)
    assert_lse_close(lse, lref, 1e-5)


def test_deterministic(fd):
    p = W.random_problem(1, 8, 8, 20000, 128, seed=6, device=DEV)
    a, la = run_dense(fd, p, seq_lens=False)
    b, lb = run_dense(fd, p, seq_lens=False)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_dominant_key_and_constant_keys(fd):
    # closed forms on the GPU path too: identical keys give the mean of V,
    # one key far above the rest gives that key's value row
    B, Hq, Hkv, L, d = 1, 4, 1, 3000, 128
    p = W.random_problem(B, Hq, Hkv, L, d, seed=8, device=DEV)
    k = p.k.clone()
    k[:] = k[:, :, :1]
    out, _ = fd.fd_decode_dense(p.q, k, p.v, None, p.scale, out_dtype="f32")
    mean = p.v.float().mean(dim=2)[0, 0]
    assert (out[0] - mean).abs().max().item() < 1e-5
    qh = W.group_direction(p.q, Hkv)[0, 0]
    k = p.k.float()
    k[0, 0, 1234] += 200.0 * qh
    out, _ = fd.fd_decode_dense(p.q, k.to(torch.bfloat16), p.v, None, p.scale, out_dtype="f32")
    assert (out[0] - p.v[0, 0, 1234].float()).abs().max().item() < 1e-4


# ------------------------------------------------------------------- paged

@pytest.mark.parametrize("identity", [True, False])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_paged_parity(fd, oracle, identity, G):
    lens = [1, 64, 65, 700, 3000, 0]
    Hkv = 2
    p = W.random_problem(len(lens), Hkv * G, Hkv, 3000, 128, seed=G, device=DEV, seq_lens=lens)
    pp = W.to_paged(p, seed=3, identity=identity, poison_tail=True)
    ref, lref = oracle.decode_paged(bits(pp.q), bits(pp.k_pages), bits(pp.v_pages), pp.page_table.cpu(),
                                    pp.num_pages, pp.seq_lens.cpu(), pp.scale)
    for ns in (0, 1, 4):
        out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens,
                                      pp.scale, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)
    # and the contiguous kernel on the same tokens gives the same answer
    out_c, _ = run_dense(fd, p, out_dtype="f32")
    out_p, _ = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens,
                                  pp.scale, out_dtype="f32")
    assert (out_c - out_p).abs().max().item() < 1e-5


def test_paged_bad_page_id_is_reported_not_read(fd, oracle):
    p = W.random_problem(2, 4, 2, 300, 128, seed=9, device=DEV, seq_lens=[300, 200])
    pp = W.to_paged(p, seed=4)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    table = pp.page_table.clone()
    table[1, 2] = pp.num_pages + 5         # out of the pool
    table[0, 0] = -3
    out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, table, pp.num_pages, pp.seq_lens, pp.scale)
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_BAD_PAGE_TABLE
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert torch.isfinite(out.float()).all()


def test_workspace_too_small_raises(fd):
    p = W.random_problem(1, 8, 2, 4096, 128, seed=10, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        fd.fd_decode_dense(p.q, p.k, p.v, None, p.scale, num_splits=4, workspace=ws)


# --------------------------------------------------------- full workloads

def sample_rows_oracle(oracle, p, heads):
    """Oracle on the given KV heads only (all sequences): returns {(b, hq): (out, lse)}."""
    G = p.Hq // p.Hkv
    res = {}
    for h in heads:
        q = bits(p.q[:, h * G:(h + 1) * G])
        k = bits(p.k[:, h:h + 1])
        v = bits(p.v[:, h:h + 1])
        o, l = oracle.decode_dense(q, k, v, p.seq_lens.cpu(), p.scale)
        for b in range(p.B):
            for g in range(G):
                res[(b, h * G + g)] = (o[b, g], l[b, g])
    return res


def check_sampled(out, lse, samples):
    for (b, hq), (o, l) in samples.items():
        assert_out_close(out[b, hq], o, BF16_TOL, what=f"out[{b},{hq}]")
        assert abs(float(lse[b, hq]) - l) <= 1e-3


def test_full_mha32k(fd, oracle):
    p = W.mha32k(seed=0, device=DEV)
    ref, lref = oracle_dense(oracle, p)
    out, lse = run_dense(fd, p, seq_lens=False)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)


def test_full_million(fd, oracle):
    p = W.million(seed=0, device=DEV)
    out, lse = run_dense(fd, p, seq_lens=False)
    check_sampled(out, lse, sample_rows_oracle(oracle, p, heads=[0, 5]))
    # the sinks carry a visible share of the attention: the LSE sits well above a plain N(0,1) field
    assert torch.isfinite(lse).all()


@pytest.mark.parametrize("B,L", [(32, 4096), (8, 32768)])
def test_ladder_batched_rungs_sampled(fd, oracle, B, L):
    # context-length ladder shapes at batch 8 and 32 (GQA-4, d=128) with the planner's chunking: every
    # sequence of two KV heads against the oracle
    p = W.ladder(B=B, L=L, seed=3, device=DEV)
    out, lse = run_dense(fd, p, seq_lens=False)
    check_sampled(out, lse, sample_rows_oracle(oracle, p, heads=[0, 7]))
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_full_gqa_paged(fd, oracle):
    pp = W.gqa_paged(seed=0, device=DEV)
    out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens,
                                  pp.scale)
    ref, lref = oracle.decode_paged(bits(pp.q), bits(pp.k_pages), bits(pp.v_pages), pp.page_table.cpu(),
                                    pp.num_pages, pp.seq_lens.cpu(), pp.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_many_short_ragged_sequences(fd, oracle):
    # thousands of sequences (grid z = B), lengths 0..200 including empty ones, planner's chunking
    B = 3000
    g = torch.Generator().manual_seed(12)
    lens = torch.randint(0, 201, (B,), generator=g).tolist()
    p = W.random_problem(B, 8, 2, 200, 64, seed=12, device=DEV, seq_lens=lens)
    ref, lref = oracle_dense(oracle, p)
    for ns in (0, 1, 3):
        out, lse = run_dense(fd, p, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)
    pp = W.to_paged(p, seed=5)
    out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens,
                                  pp.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
