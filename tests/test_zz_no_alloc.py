"""fd_decode_dense_noalloc: the dense decode for callers that cannot allocate
device memory (a plug-in inside a host engine that owns all device memory,
or a loop that must not call cudaMalloc because it can synchronise the
device).  Its scratch is a fixed array inside the library.

Checked through the C ABI against fd_decode_dense and against the CPU
oracle on calls in a row: first a long call with many chunks that fills much
of the array, then a ragged call whose short sequence has empty chunks (the
merge must not read the stale partials the first call left there), then a
one-chunk call (no scratch at all); plus the size limit.  Collected last, so
a failure here comes after every other test.
"""
import pytest
import torch

import workloads as W
from parity import BF16_TOL, F32_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu


def reference(fd, p, out_dtype, num_splits):
    return fd.fd_decode_dense(p.q, p.k, p.v, p.seq_lens, p.scale, num_splits=num_splits,
                              out_dtype=out_dtype)


def noalloc(fd, p, out_dtype, num_splits):
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.empty((p.B, p.Hq, p.d), dtype=dt, device=p.q.device)
    lse = torch.empty((p.B, p.Hq), dtype=torch.float32, device=p.q.device)
    return fd.fd_decode_dense_noalloc(p.q, p.k, p.v, out, p.seq_lens, p.scale, num_splits=num_splits,
                                      lse=lse)


def test_noalloc_matches_dense_and_oracle_on_calls_in_a_row(fd, oracle):
    # 64 chunks x 32 query heads x 130 floats ~ 1.1 MB of partials, then a ragged batch of
    # 40 chunks per sequence in which the 777-token sequence fills only 13 of them
    first = W.random_problem(1, 32, 8, 64 * 1024, 128, seed=20, device="cuda")
    second = W.random_problem(2, 16, 4, 20000, 128, seed=21, device="cuda", seq_lens=[20000, 777])
    third = W.random_problem(1, 8, 8, 9000, 64, seed=22, device="cuda")
    cases = [(first, "bf16", 64, BF16_TOL), (second, "bf16", 40, BF16_TOL), (third, "f32", 1, F32_TOL),
             (second, "f32", 0, F32_TOL)]
    assert fd.fd_decode_workspace_size(1, 32, 8, 64 * 1024, 128, 64, False) > \
        fd.fd_decode_workspace_size(2, 16, 4, 20000, 128, 40, True)
    assert fd.fd_decode_workspace_size(1, 8, 8, 9000, 64, 1, False) == 0
    for p, dt, ns, tol in cases:
        out, lse = noalloc(fd, p, dt, ns)
        ref, lref = reference(fd, p, dt, ns)
        torch.cuda.synchronize()
        assert_out_close(out, ref.double().cpu().numpy(), tol)
        assert_lse_close(lse, lref.double().cpu().numpy())
        oref, olse = oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)
        assert_out_close(out, oref, tol)
        assert_lse_close(lse, olse)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_noalloc_rejects_plans_beyond_its_scratch(fd):
    # 64 query heads x 1000 chunks x (128 + 2) floats > 4 MiB
    p = W.random_problem(1, 64, 8, 64000, 128, seed=23, device="cuda")
    out = torch.empty((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fd.FdError) as e:
        fd.fd_decode_dense_noalloc(p.q, p.k, p.v, out, None, p.scale, num_splits=1000)
    assert e.value.status == fd.FD_ERR_WORKSPACE_TOO_SMALL
