"""Tolerances and comparison helpers for GPU-vs-oracle parity.

bf16 workloads: max-abs error 1.5e-2 and mean-abs error 2e-3 on O; f32
workloads: max-abs 1e-4 on O; LSE within 1e-3 relative for both."""
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
