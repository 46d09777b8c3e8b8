"""Shared helpers for the GPU-vs-oracle parity tests (no method arithmetic)."""
import numpy as np
import torch

# Tolerances.  bf16 outputs: max|err| <= 1e-2 * (1 + |ref|), per element.
# fp32 outputs: the kernel accumulates in fp32 with a 2^x approximation of
# relative error ~2^-22, so 1e-4 * (1 + |ref|) leaves two orders of margin.
# LSE: 1e-3 absolute.
BF16_TOL = 1e-2
F32_TOL = 1e-4
LSE_TOL = 1e-3


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_out_close(got, ref, tol, what="out"):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bound = tol * (1.0 + np.abs(ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: max excess at {worst}: got {g[worst]}, ref {ref[worst]}, err {err[worst]}"
    return float(err.max())


def assert_lse_close(got, ref, tol=LSE_TOL):
    g = got.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), inf_ref), "lse: -inf pattern differs"
    err = np.abs(g[~inf_ref] - ref[~inf_ref])
    assert err.size == 0 or err.max() <= tol, f"lse: max err {err.max()}"
    return float(err.max()) if err.size else 0.0
