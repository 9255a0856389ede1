"""Pins for the backward oracle (CPU only): finite differences of the
forward oracle, autograd through a dense masked formulation, and special
cases the structure fixes."""
import math

import numpy as np
import pytest

from oracle import tree_attention as ta
from oracle import tree_backward as tb
from tree_structured_shared_gb300 import workloads as wl

from test_oracle import _dense_mask


def _case(seed, order=ta.PACK_CANONICAL, Hq=4, Hkv=2, d=8, **kw):
    w = wl.random_pages(seed, allow_empty=False, Hq=Hq, Hkv=Hkv, d=d, **kw)
    T = w.n_tokens
    q = wl.normal_f32(seed * 7 + 1, (T, Hq, d))
    k = wl.normal_f32(seed * 7 + 2, (T, Hkv, d))
    v = wl.normal_f32(seed * 7 + 3, (T, Hkv, d))
    dO = wl.normal_f32(seed * 7 + 4, (T, Hq, d))
    return w, q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), dO.astype(np.float64)


def test_finite_differences():
    """Central differences of L = sum(dO * O) through the forward oracle at
    sampled coordinates of q, k and v."""
    w, q, k, v, dO = _case(3, n_pages=2, max_prefix=6, max_regions=3, max_layout=3, max_content=5)
    dQ, dK, dV = tb.tree_backward(q, k, v, dO, w.pages)
    rng = np.random.default_rng(0)
    h = 1e-6

    def loss(q_, k_, v_):
        O, _ = ta.tree_forward(q_, k_, v_, w.pages)
        return float((O * dO).sum())

    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for _ in range(25):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("order", [ta.PACK_CANONICAL, ta.PACK_DOCUMENT])
def test_dense_autograd(seed, order):
    """torch autograd through dense masked attention, the mask written as
    region comparisons (a formulation separate from the ancestor lists)."""
    torch = pytest.importorskip("torch")
    w, q, k, v, dO = _case(10 + seed, order, n_pages=3, max_prefix=10, max_regions=4, max_layout=4,
                           max_content=7)
    dQ, dK, dV = tb.tree_backward(q, k, v, dO, w.pages, order)
    mask = torch.from_numpy(_dense_mask(w.pages, order))
    G = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    s = torch.einsum("qhd,khd->hqk", tq, tk.repeat_interleave(G, dim=1)) / math.sqrt(q.shape[2])
    s = s.masked_fill(~mask[None], float("-inf"))
    o = torch.einsum("hqk,khd->qhd", torch.softmax(s, dim=2), tv.repeat_interleave(G, dim=1))
    (o * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-11, rtol=0)


def test_special_cases():
    """The first prefix token sees only itself: its softmax is constant, so
    dq = 0 there.  The last token of a content branch is seen by itself
    only: dV there is P_tt * dO_t summed over the group's heads, with P_tt
    from the forward's LSE."""
    w, q, k, v, dO = _case(21, n_pages=1, max_prefix=8, max_regions=3, max_layout=3, max_content=6)
    pg = w.pages[0]
    dQ, dK, dV = tb.tree_backward(q, k, v, dO, w.pages)
    assert np.all(dQ[0] == 0.0)
    O, L = ta.tree_forward(q, k, v, w.pages)
    t = w.n_tokens - 1  # last token of the last content branch in canonical packing
    Hq, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    G = Hq // Hkv
    for g in range(Hkv):
        want = np.zeros(d)
        for h in range(g * G, (g + 1) * G):
            p = math.exp(q[t, h] @ k[t, g] / math.sqrt(d) - L[h, t])
            want += p * dO[t, h]
        np.testing.assert_allclose(dV[t, g], want, atol=1e-13)
    assert pg.content_len[-1] >= 1


def test_isolation():
    """An upstream gradient on the tokens of one content branch Y_j only
    reaches dQ of Y_j and dK/dV of Y_j's ancestors (X, B<=j, Y_j)."""
    w, q, k, v, dO = _case(5, n_pages=1, max_prefix=6, max_regions=4, max_layout=3, max_content=5)
    ident, pos = ta.packed_layout(w.pages)
    N = len(w.pages[0].layout_len)
    j = N - 2 if N >= 2 else 0
    in_yj = np.array([(kind == ta.Y_KIND and r == j) for (_, kind, r, _) in ident])
    anc = np.array([kind == ta.X_KIND or (kind == ta.B_KIND and r <= j) or (kind == ta.Y_KIND and r == j)
                    for (_, kind, r, _) in ident])
    dO = np.where(in_yj[:, None, None], dO, 0.0)
    dQ, dK, dV = tb.tree_backward(q, k, v, dO, w.pages)
    assert np.all(dQ[~in_yj] == 0)
    assert np.all(dK[~anc] == 0) and np.all(dV[~anc] == 0)
    assert np.abs(dV[anc]).sum() > 0


def test_restricted_positions_match_full():
    """Restricting the query positions reproduces the full result on those
    rows, and on keys that only those queries see."""
    w, q, k, v, dO = _case(8, n_pages=2, max_prefix=6, max_regions=3, max_layout=3, max_content=6)
    full = tb.tree_backward(q, k, v, dO, w.pages)
    ident, _ = ta.packed_layout(w.pages)
    # the last content region of page 0: its keys are seen by its own tokens only
    p0 = w.pages[0]
    N = len(p0.layout_len)
    rows = [t for t, (p, kind, r, _) in enumerate(ident) if p == 0 and kind == ta.Y_KIND and r == N - 1]
    part = tb.tree_backward(q, k, v, dO, w.pages, positions=rows)
    np.testing.assert_allclose(part[0][rows], full[0][rows], atol=1e-13, rtol=0)
    np.testing.assert_allclose(part[1][rows], full[1][rows], atol=1e-13, rtol=0)
    np.testing.assert_allclose(part[2][rows], full[2][rows], atol=1e-13, rtol=0)
