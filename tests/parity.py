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


# ---------------------------------------------------------------- pooled oracle
# Whole-page oracle runs at full size take minutes of float64 work, so the
# rows are dealt out to a pool of spawned processes (spawn, not fork: the
# parent has already used the GPU).  Each worker memory-maps the inputs from
# an .npz written by the test and runs the oracle on its rows only.


def _load(path):
    z = np.load(path)
    return {k: z[k] for k in z.files}


def _forward_rows(args):
    path, pages, rows = args
    from oracle import tree_attention as ta
    x = _load(path)
    O, L = ta.tree_forward(x["q"], x["k"], x["v"], pages, positions=rows)
    return rows, O[rows], L[:, rows]


def _backward_rows(args):
    path, pages, rows = args
    from oracle import tree_backward as tb
    x = _load(path)
    dQ, dK, dV = tb.tree_backward(x["q"], x["k"], x["v"], x["do"], pages, positions=rows)
    return rows, dQ[rows], dK, dV


def _pool_map(fn, path, pages, rows, n_chunks):
    import multiprocessing as mp
    import os
    rows = list(rows)
    n_proc = max(1, min(len(os.sched_getaffinity(0)), n_chunks))
    chunks = [rows[c::n_chunks] for c in range(n_chunks) if rows[c::n_chunks]]
    with mp.get_context("spawn").Pool(processes=n_proc) as pool:
        return pool.map(fn, [(path, pages, sorted(c)) for c in chunks])


def pooled_forward(path, pages, T, Hq, d, rows=None, n_chunks=64):
    """The oracle's forward O [T, Hq, d] and LSE [Hq, T] over `rows` (all by
    default; other rows stay NaN), computed by a process pool."""
    rows = range(T) if rows is None else rows
    O = np.full((T, Hq, d), np.nan)
    L = np.full((Hq, T), np.nan)
    for r, o, l in _pool_map(_forward_rows, path, pages, rows, n_chunks):
        O[r] = o
        L[:, r] = l
    return O, L


def pooled_backward(path, pages, T, Hq, Hkv, d, rows=None, n_chunks=64):
    """The oracle's dQ (on `rows`), dK and dV (the contributions of those
    rows: the whole gradient of every key that only they see), computed by a
    process pool; the chunks' key gradients add."""
    rows = range(T) if rows is None else rows
    dQ = np.full((T, Hq, d), np.nan)
    dK = np.zeros((T, Hkv, d))
    dV = np.zeros((T, Hkv, d))
    for r, dq, dk, dv in _pool_map(_backward_rows, path, pages, rows, n_chunks):
        dQ[r] = dq
        dK += dk
        dV += dv
    return dQ, dK, dV
