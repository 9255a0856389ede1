"""Tree-varlen backward on the GPU against the float64 oracle."""
import numpy as np
import pytest

from oracle import tree_backward as tb
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check_grad

pytestmark = pytest.mark.gpu


def _run(w, seed, order=padoc.PACK_CANONICAL):
    import torch
    from tree_structured_shared_gb300 import harness
    q, k, v = wl.tree_qkv(w, seed)
    d_o = wl.normal_f32(seed * 3 + 7, (w.n_tokens, w.Hq, w.d), w.value_scale)
    if w.dtype == "bf16":
        d_o = wl.round_bf16(d_o)
    f = harness.Forward(w, q, k, v, order)
    f.run()
    b = harness.Backward(f, d_o)
    dq, dk, dv = b.run()
    torch.cuda.synchronize()
    padoc.device_status()
    ref = tb.tree_backward(q, k, v, d_o, w.pages, order)
    got = [x.float().cpu().numpy() for x in (dq, dk, dv)]
    return got, ref, b


def test_tiny_f32_page(padoc_lib):
    w = wl.tiny_fp32_page(0)
    got, ref, _ = _run(w, 0)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        check_grad(g, r, "f32", name)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("order", [padoc.PACK_CANONICAL, padoc.PACK_DOCUMENT])
def test_random_pages_bf16(padoc_lib, seed, order):
    w = wl.random_pages(40 + seed, n_pages=3, max_prefix=300, max_regions=5, max_layout=20, max_content=150,
                        Hq=4, Hkv=2, d=128, dtype="bf16")
    got, ref, _ = _run(w, seed, order)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        check_grad(g, r, "bf16", f"{name} seed {seed} order {order}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_groups(padoc_lib, G):
    w = wl.random_pages(60 + G, n_pages=2, max_prefix=200, max_regions=4, max_layout=12, max_content=120,
                        allow_empty=False, Hq=2 * G, Hkv=2, d=128, dtype="bf16")
    got, ref, _ = _run(w, G)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        check_grad(g, r, "bf16", f"{name} G={G}")


def test_deterministic(padoc_lib):
    import torch
    w = wl.random_pages(70, n_pages=2, max_prefix=400, max_regions=4, max_layout=12, max_content=200,
                        allow_empty=False, Hq=4, Hkv=2, d=128, dtype="bf16")
    _, _, b = _run(w, 1)
    first = [x.clone() for x in (b.dq, b.dk, b.dv)]
    b.run()
    torch.cuda.synchronize()
    for a, c in zip(first, (b.dq, b.dk, b.dv)):
        assert torch.equal(a, c)


def test_cuda_core_path_bf16(padoc_lib, tmp_path):
    """The CUDA-core kernels (selected by PADOC_BWD_CORE=1) on a bf16 case
    the tensor-core path also serves; run in a child process because the
    switch is read once per process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = tmp_path / "grads.npz"
    code = (
        "import sys, numpy as np, torch; sys.path.insert(0, %r)\n"
        "from tree_structured_shared_gb300 import harness, workloads as wl\n"
        "w = wl.random_pages(81, n_pages=2, max_prefix=200, max_regions=4, max_layout=12, max_content=120,"
        " allow_empty=False, Hq=4, Hkv=2, d=128, dtype='bf16')\n"
        "q, k, v = wl.tree_qkv(w, 2)\n"
        "d_o = wl.round_bf16(wl.normal_f32(13, (w.n_tokens, 4, 128), w.value_scale))\n"
        "f = harness.Forward(w, q, k, v); f.run(); b = harness.Backward(f, d_o); b.run(); torch.cuda.synchronize()\n"
        "np.savez(%r, *[x.float().cpu().numpy() for x in (b.dq, b.dk, b.dv)])\n"
    ) % (root, str(out))
    env = dict(os.environ, PADOC_BWD_CORE="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    w = wl.random_pages(81, n_pages=2, max_prefix=200, max_regions=4, max_layout=12, max_content=120,
                        allow_empty=False, Hq=4, Hkv=2, d=128, dtype="bf16")
    q, k, v = wl.tree_qkv(w, 2)
    d_o = wl.round_bf16(wl.normal_f32(13, (w.n_tokens, 4, 128), w.value_scale))
    ref = tb.tree_backward(q, k, v, d_o, w.pages)
    for i, name in enumerate(("dq", "dk", "dv")):
        check_grad(got[f"arr_{i}"], ref[i], "bf16", f"core {name}")


def test_packed_backward_sampled_regions(padoc_lib):
    """The bench's training workload, 8 packed sequences of 16384 tokens, in
    one backward launch; checked on the tokens of sampled content regions.
    A content token's key is seen only by later tokens of its own region, so
    the oracle restricted to those queries gives their dQ, dK and dV."""
    import torch
    from oracle import tree_attention as ta
    from tree_structured_shared_gb300 import harness
    fw = wl.packed_sequences(0)
    f = harness.Forward(fw, seed=0)
    f.run()
    b = harness.Backward(f, seed=0)
    b.run()
    torch.cuda.synchronize()
    padoc.device_status()
    starts = np.cumsum([0] + [p.n_tokens for p in fw.pages])
    with_content = [i for i, pg in enumerate(fw.pages) if any(c > 0 for c in pg.content_len)]
    for pi in [with_content[1], with_content[len(with_content) // 2], with_content[-1]]:
        a, e = int(starts[pi]), int(starts[pi + 1])
        page = [fw.pages[pi]]
        ident, _ = ta.packed_layout(page)
        N = len(page[0].layout_len)
        regions = [r for r in range(N) if page[0].content_len[r] > 0]
        for r in (regions[0], regions[-1]):
            rows = [t for t, (_, kind, rr, _) in enumerate(ident) if kind == ta.Y_KIND and rr == r]
            host = [x[a:e].float().cpu().numpy() for x in (f.q, f.k, f.v, b.d_o)]
            ref = tb.tree_backward(*host, page, positions=rows)
            for g, rr_, name in zip((b.dq, b.dk, b.dv), ref, ("dq", "dk", "dv")):
                check_grad(g[a:e].float().cpu().numpy()[rows], rr_[rows], "bf16", f"page {pi} region {r} {name}")


def test_packed_backward_whole_page(padoc_lib, tmp_path):
    """The bench's training workload (8 packed sequences of 16384 tokens) in
    one backward launch, checked on one whole page: the smallest page that
    has a prefix, layout and content.  Only a page's own queries see its
    keys, so the oracle over every query of the page gives every gradient on
    it, including dK / dV of the prefix keys, which the key-stationary pass
    accumulates over thousands of queries in dozens of query tiles."""
    import torch
    from oracle import tree_attention as ta
    from parity import pooled_backward
    from tree_structured_shared_gb300 import harness
    fw = wl.packed_sequences(0)
    f = harness.Forward(fw, seed=0)
    f.run()
    b = harness.Backward(f, seed=0)
    b.run()
    torch.cuda.synchronize()
    padoc.device_status()
    starts = np.cumsum([0] + [p.n_tokens for p in fw.pages])
    cand = [i for i, pg in enumerate(fw.pages) if sum(pg.layout_len) > 0 and sum(pg.content_len) > 0]
    pi = min(cand, key=lambda i: fw.pages[i].n_tokens)
    a, e = int(starts[pi]), int(starts[pi + 1])
    page = [fw.pages[pi]]
    T = e - a
    assert fw.pages[pi].prefix_len >= 4000 and T >= 4000
    host = [x[a:e].float().cpu().numpy() for x in (f.q, f.k, f.v, b.d_o)]
    path = str(tmp_path / "page.npz")
    np.savez(path, q=host[0], k=host[1], v=host[2], do=host[3])
    dQ, dK, dV = pooled_backward(path, page, T, fw.Hq, fw.Hkv, fw.d)
    got = [g[a:e].float().cpu().numpy() for g in (b.dq, b.dk, b.dv)]
    ident, _ = ta.packed_layout(page)
    X = [t for t, x in enumerate(ident) if x[1] == ta.X_KIND]
    B = [t for t, x in enumerate(ident) if x[1] == ta.B_KIND]
    assert len(X) >= 4000 and len(B) > 0
    check_grad(got[0], dQ, "bf16", f"page {pi} dq (all {T} rows)")
    for g, r, name in ((got[1], dK, "dk"), (got[2], dV, "dv")):
        check_grad(g, r, "bf16", f"page {pi} {name} (all keys)")
        check_grad(g[X], r[X], "bf16", f"page {pi} {name} (prefix keys)")
        check_grad(g[B], r[B], "bf16", f"page {pi} {name} (layout keys)")

