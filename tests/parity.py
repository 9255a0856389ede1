"""Tolerances and comparison helpers for GPU-vs-oracle parity.

bf16 workloads: max-abs error 1.5e-2 and mean-abs error 2e-3 on O; f32
workloads: max-abs 1e-4 on O; LSE within 1e-3 relative for both.

Backward gradients are compared relative to their own scale (their
magnitudes grow with the number of queries that see a key): bf16 max error
within 1e-2 of max|ref| and mean error within 5e-3 of mean|ref| (output
rounding alone is 2^-9 relative; bf16 probabilities in the tensor-core path
add the same order per term); f32 within 1e-4 and 1e-5."""
import numpy as np

BF16_MAX_ABS, BF16_MEAN_ABS = 1.5e-2, 2e-3
F32_MAX_ABS = 1e-4
LSE_REL = 1e-3


def check(o_gpu, lse_gpu, o_ref, lse_ref, dtype="bf16", what=""):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    err = np.abs(o_gpu - o_ref)
    if dtype == "bf16":
        assert err.max() <= BF16_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    else:
        assert err.max() <= F32_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    lg = np.asarray(lse_gpu, np.float64)
    lr = np.asarray(lse_ref, np.float64)
    rel = np.abs(lg - lr) / np.maximum(np.abs(lr), 1e-6)
    assert rel.max() <= LSE_REL, f"{what}: LSE rel {rel.max():.3e}"
    return float(err.max()), float(err.mean()), float(rel.max())


GRAD_BF16_MAX, GRAD_BF16_MEAN = 1e-2, 5e-3
GRAD_F32_MAX, GRAD_F32_MEAN = 1e-4, 1e-5


def check_grad(g_gpu, g_ref, dtype="bf16", what=""):
    g = np.asarray(g_gpu, np.float64)
    r = np.asarray(g_ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    err = np.abs(g - r)
    rmax = err.max() / max(np.abs(r).max(), 1e-30)
    rmean = err.mean() / max(np.abs(r).mean(), 1e-30)
    lim = (GRAD_BF16_MAX, GRAD_BF16_MEAN) if dtype == "bf16" else (GRAD_F32_MAX, GRAD_F32_MEAN)
    assert rmax <= lim[0], f"{what}: max error {rmax:.3e} of max|ref|"
    assert rmean <= lim[1], f"{what}: mean error {rmean:.3e} of mean|ref|"
    return float(rmax), float(rmean)
