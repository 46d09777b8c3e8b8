"""GPU parity of the unified-max variant (FlashDecoding++ summary, sections
1, 3 and 5: one fixed max value phi for every chunk, with a fallback to the
running maximum when the scores leave the range where that is exact).

The oracle is the unchanged binary64 definition of attention: the variant
must reach the same result for every phi.  The cases cover a phi above every
score (the fixed-reference path throughout), a phi below the scores and one
far above them (the fallback at the first tile), and one dominant key far
above phi in the middle of a long chunk (the fallback after many tiles on
the reference).  That each path was taken is read from the chunk maxima m_i
the partial pass leaves in the workspace ([B, Hq, S, D] partial outputs, then
[B, Hq, S, 2] pairs (m_i in log2 units, l_i)).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from parity import BF16_TOL, F32_TOL, assert_lse_close, assert_out_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
LOG2E = 1.4426950408889634


def oracle_ref(oracle, p):
    return oracle.decode_dense(bits(p.q), bits(p.k), bits(p.v), p.seq_lens.cpu(), p.scale)


def chunk_maxima(fd, p, phi, num_splits, out_dtype="f32"):
    """Runs the unified variant with an explicit workspace; returns out, lse
    and the per-chunk maxima m_i [B, Hq, S] (log2 units)."""
    ragged = p.seq_lens is not None
    S = fd.fd_num_splits(p.B, p.Hq, p.Hkv, p.L_max, p.d, num_splits, ragged)
    need = fd.fd_decode_workspace_size(p.B, p.Hq, p.Hkv, p.L_max, p.d, num_splits, ragged)
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device=DEV)
    out, lse = fd.fd_decode_dense_unified(p.q, p.k, p.v, p.seq_lens, p.scale, phi, num_splits, out_dtype=out_dtype,
                                          workspace=ws)
    torch.cuda.synchronize()
    ml = ws[p.B * p.Hq * S * p.d:p.B * p.Hq * S * p.d + p.B * p.Hq * S * 2].view(p.B, p.Hq, S, 2)
    return out, lse, ml[..., 0].cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("phi", [6.5, 0.0, 100.0, -100.0])
def test_unified_parity_small(fd, oracle, d, G, phi):
    lens = [1, 63, 64, 65, 1000, 4100]
    Hkv = 2
    p = W.random_problem(len(lens), Hkv * G, Hkv, 4100, d, seed=7 * G + d, device=DEV, seq_lens=lens)
    ref, lref = oracle_ref(oracle, p)
    for ns in (0, 1, 3, 8):
        for dt, tol in (("bf16", BF16_TOL), ("f32", F32_TOL)):
            out, lse = fd.fd_decode_dense_unified(p.q, p.k, p.v, p.seq_lens, p.scale, phi, ns, out_dtype=dt)
            torch.cuda.synchronize()
            assert_out_close(out, ref, tol, what=f"ns={ns} {dt}")
            assert_lse_close(lse, lref)


def test_unified_empty_sequences(fd, oracle):
    p = W.random_problem(3, 8, 2, 300, 128, seed=3, device=DEV, seq_lens=[0, 300, 0])
    out, lse = fd.fd_decode_dense_unified(p.q, p.k, p.v, p.seq_lens, p.scale, 6.5, 2, out_dtype="f32")
    ref, lref = oracle_ref(oracle, p)
    assert_out_close(out, ref, F32_TOL)
    assert_lse_close(lse, lref)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[2]))


@pytest.mark.parametrize("G", [1, 4])
def test_unified_reference_path_and_both_fallbacks(fd, oracle, G):
    """phi above every score: every chunk reports m_i = phi (no maximum was
    taken); phi far above or below the scores: every chunk falls back and
    reports its true maximum."""
    p = W.random_problem(1, 2 * G, 2, 8192, 128, seed=11 + G, device=DEV)
    ref, lref = oracle_ref(oracle, p)
    smax = float(p.scale * (p.q.double().view(1, 2, G, 128) @ p.k.double()[0].transpose(-1, -2)).max())
    assert smax < 8.0
    for phi, on_reference in ((8.0, True), (-100.0, False), (200.0, False)):
        out, lse, m = chunk_maxima(fd, p, phi, 4)
        assert_out_close(out, ref, F32_TOL)
        assert_lse_close(lse, lref)
        if on_reference:
            np.testing.assert_array_equal(m, np.float32(np.float32(phi) * np.float32(LOG2E)))
        else:
            assert np.all(m < smax * LOG2E + 1e-3) and np.all(m > (smax - 10) * LOG2E)


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("out_dtype,tol", [("bf16", BF16_TOL), ("f32", F32_TOL)])
def test_unified_dominant_key_far_above_phi(fd, oracle, G, out_dtype, tol):
    """One key whose score is ~40 nats above phi, 5000 tokens into a chunk of
    8192: the chunk runs ~78 tiles on the reference, then rebases; the output
    is (almost exactly) that key's value row."""
    L = 16384
    p = W.random_problem(1, G, 1, L, 128, seed=5, device=DEV)
    qd = p.q[0].float()
    u = qd.sum(0)
    qh = u / u.norm()
    j = 5000
    c = (40.0 + 6.5) / (p.scale * float((qd @ qh).min())) + 1.0
    k = p.k.clone()
    k[0, 0, j] = (k[0, 0, j].float() + c * qh).to(torch.bfloat16)
    p = W.Problem(p.name, p.q, k, p.v, p.seq_lens, p.scale, L)
    s = p.scale * (p.q[0].double() @ p.k[0, 0].double().T)
    assert float(s[:, j].min()) > 6.5 + 40 and float(np.delete(s.cpu().numpy(), j, axis=1).max()) < 6.5
    ref, lref = oracle_ref(oracle, p)
    out, lse, m = chunk_maxima(fd, p, 6.5, 2, out_dtype)
    assert_out_close(out, ref, tol)
    assert_lse_close(lse, lref)
    phi2 = np.float32(np.float32(6.5) * np.float32(LOG2E))
    assert np.all(m[0, :, 0] > phi2 + 40)        # the chunk with the key fell back
    np.testing.assert_array_equal(m[0, :, 1], phi2)  # the other stayed on phi


def test_unified_paged(fd, oracle):
    p = W.random_problem(3, 16, 2, 3000, 128, seed=13, device=DEV, seq_lens=[3000, 1, 2345])
    pp = W.to_paged(p, seed=4)
    ref, lref = oracle_ref(oracle, p)
    for phi in (6.5, -50.0):
        out, lse = fd.fd_decode_paged_unified(pp.q, pp.k_pages, pp.v_pages, pp.page_table, pp.num_pages,
                                              pp.seq_lens, pp.scale, phi, out_dtype="f32")
        torch.cuda.synchronize()
        assert_out_close(out, ref, F32_TOL)
        assert_lse_close(lse, lref)
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_unified_full_million_sampled(fd, oracle):
    """The 1M-token workload in the benchmark's launch configuration, phi = 6.5
    (every score of this workload lies below it); oracle on two KV heads."""
    p = W.million(seed=0, device=DEV)
    out, lse = fd.fd_decode_dense_unified(p.q, p.k, p.v, None, p.scale, 6.5)
    torch.cuda.synchronize()
    G = p.Hq // p.Hkv
    for h in (0, 5):
        ref, lref = oracle.decode_dense(bits(p.q[:, h * G:(h + 1) * G]), bits(p.k[:, h:h + 1]),
                                        bits(p.v[:, h:h + 1]), None, p.scale)
        assert_out_close(out[:, h * G:(h + 1) * G], ref, BF16_TOL)
        assert_lse_close(lse[:, h * G:(h + 1) * G], lref)
