"""GPU parity at the GQA group sizes the other suites skip (2, 5, 6, 7 query
heads per KV head), for every cache kind: the tensor-core consumers pad the
group to 8 columns, so these sizes move the boundary between real and padded
columns inside and across the lanes' column pairs.  Each case is compared with
the oracle: bf16 and the narrow caches as attention over the (decoded) rows,
top-delta with its selection sets."""
import pytest
import torch

import workloads as W
from parity import BF16_TOL, assert_lse_close, assert_out_close, bits
from test_gpu_topdelta import check_topdelta, run_both

pytestmark = pytest.mark.gpu

DEV = "cuda"
GROUPS = [2, 5, 6, 7]


def problem(G, d, seed):
    lens = [1500, 0, 777]
    return W.random_problem(len(lens), 2 * G, 2, 1500, d, seed=seed, device=DEV, seq_lens=lens)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", GROUPS)
def test_bf16_group_sizes(fd, oracle, G, d):
    p = problem(G, d, 40 + G)
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)
    for ns in (0, 3):
        out, lse = fd.fd_decode_dense(p.q, p.k, p.v, p.seq_lens, p.scale, num_splits=ns)
        assert_out_close(out, ref, BF16_TOL)
        assert_lse_close(lse, lref)


@pytest.mark.parametrize("G", GROUPS)
def test_fp8_group_sizes(fd, oracle, G):
    p = problem(G, 128, 50 + G)
    sl = p.seq_lens.cpu()
    kc, ks = oracle.quantize_kv_fp8(bits(p.k), sl)
    vc, vs = oracle.quantize_kv_fp8(bits(p.v), sl)
    ref, lref = oracle.decode_dense_fp8(bits(p.q), kc, ks, vc, vs, sl, p.scale)
    dev = [torch.from_numpy(a).to(DEV) for a in (kc, ks, vc, vs)]
    out, lse = fd.fd_decode_dense_fp8(p.q, *dev, p.seq_lens, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("G", GROUPS)
def test_fp4_group_sizes(fd, oracle, G):
    p = problem(G, 128, 60 + G)
    sl = p.seq_lens.cpu()
    kc, ks = oracle.quantize_kv_fp4(bits(p.k), sl)
    vc, vs = oracle.quantize_v_fp4(bits(p.v), sl)
    ref, lref = oracle.decode_dense_fp4(bits(p.q), kc, ks, vc, vs, sl, p.scale)
    dev = [torch.from_numpy(a).to(DEV) for a in (kc, ks, vc, vs)]
    out, lse = fd.fd_decode_dense_fp4(p.q, *dev, p.seq_lens, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("G", GROUPS)
def test_topdelta_group_sizes(fd, oracle, G):
    p = W.ffd(seed=70 + G, B=2, L=2500, Hq=2 * G, Hkv=2, d=128)
    p = W.Problem(p.name, p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.seq_lens.to(DEV), p.scale, p.L_max)
    for union in (False, True):
        enc, ref, out, lse, mask, cnt = run_both(fd, oracle, p, 5.0, group_union=union)
        check_topdelta(oracle, p, enc, ref, out, lse, mask, cnt, 5.0, BF16_TOL, group_union=union)


@pytest.mark.parametrize("G", GROUPS)
def test_paged_and_unified_group_sizes(fd, oracle, G):
    # the paged pass (tail rows of the last pages poisoned with NaN) and the fixed-max variant
    p = problem(G, 128, 80 + G)
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)
    pp = W.to_paged(p, seed=G)
    out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens, pp.scale)
    assert_out_close(out, ref, BF16_TOL, what="paged")
    assert_lse_close(lse, lref)
    for phi in (6.5, -100.0):
        out, lse = fd.fd_decode_dense_unified(p.q, p.k, p.v, p.seq_lens, p.scale, phi)
        assert_out_close(out, ref, BF16_TOL, what=f"unified phi={phi}")
        assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
