"""The time-out path of the pipeline waits, exercised without faulting the GPU.

A test-only hook (fd_debug_inject_wait_timeout) shortens every wait of the
bf16 dense/paged pass to 1 ms and makes the producer withhold one tile of
every chunk: no copy and no arrival for it, so nothing is in flight for that
stage.  The consumers' wait for the tile runs out; the kernel records
FD_ERR_DEVICE_TIMEOUT, lets the copies it did start land and returns.  The
tests check that the call returns promptly, that the status is reported, and
that the device still answers: a normal call afterwards matches the oracle.
A 1 ms limit without a withheld tile must not fire at all.
"""
import time

import pytest
import torch

import workloads as W
from parity import BF16_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu


def check_normal_call(fd, oracle, p, num_splits):
    out, lse = fd.fd_decode_dense(p.q, p.k, p.v, None, p.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("num_splits,tile", [(1, 0), (1, 5), (3, 2)])
def test_withheld_tile_times_out_and_is_reported(fd, oracle, G, num_splits, tile):
    p = W.random_problem(1, 2 * G, 2, 64 * 12, 128, seed=40 + G, device="cuda")
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    try:
        fd.fd_debug_inject_wait_timeout(1_000_000, tile)
        t0 = time.time()
        fd.fd_decode_dense(p.q, p.k, p.v, None, p.scale, num_splits=num_splits)
        status = fd.fd_device_status(clear=True)
        elapsed = time.time() - t0
    finally:
        fd.fd_debug_inject_wait_timeout(0, -1)
    assert status == fd.FD_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, elapsed
    check_normal_call(fd, oracle, p, num_splits)


def test_withheld_page_in_the_paged_pass(fd, oracle):
    p = W.random_problem(2, 8, 2, 64 * 10, 128, seed=44, device="cuda", seq_lens=[640, 300])
    pp = W.to_paged(p, seed=5)
    try:
        fd.fd_debug_inject_wait_timeout(1_000_000, 3)
        fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens, pp.scale)
        status = fd.fd_device_status(clear=True)
    finally:
        fd.fd_debug_inject_wait_timeout(0, -1)
    assert status == fd.FD_ERR_DEVICE_TIMEOUT
    out, lse = fd.fd_decode_paged(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages, pp.seq_lens,
                                  pp.scale)
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_short_limit_alone_does_not_fire(fd, oracle):
    p = W.random_problem(1, 32, 8, 1 << 16, 128, seed=45, device="cuda")
    try:
        fd.fd_debug_inject_wait_timeout(1_000_000, -1)
        for _ in range(3):
            out, lse = fd.fd_decode_dense(p.q, p.k, p.v, None, p.scale)
        status = fd.fd_device_status(clear=True)
    finally:
        fd.fd_debug_inject_wait_timeout(0, -1)
    assert status == fd.FD_OK
    ref, lref = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), None, p.scale)
    assert_out_close(out, ref, BF16_TOL)
    assert_lse_close(lse, lref)
