"""Parity at the full benchmark sizes, in the launch configuration bench.py
times (planned decode: prefix pass then own pass; forward over all packed
sequences).  Outputs are checked on sampled pages / rows that the float64
oracle computes one by one.  Inputs come from the seeded device generator
(torch's CUDA RNG, per item), copied to the host; nothing the oracle sees
comes from the CUDA path under test."""
import numpy as np
import pytest

from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def harness(padoc_lib):
    from tree_structured_shared_gb300 import harness as h
    return h


def _decode_sampled(harness, w, tree, pages):
    import torch
    d = harness.Decode(w, seed=0, tree=tree)
    d.plan()
    d.prefix_pass()
    d.own_pass()
    torch.cuda.synchronize()
    padoc.device_status()
    q_host = d.q.float().cpu().numpy()
    kn_host = d.k_new.float().cpu().numpy()
    vn_host = d.v_new.float().cpu().numpy()
    o = d.o.float().cpu().numpy()
    lse = d.lse.cpu().numpy()
    qoff = [0]
    for pg in w.pages:
        qoff.append(qoff[-1] + sum(pg.q_len))
    for p in pages:
        pg = w.pages[p]
        hv = d.host_values(p)
        rows = slice(qoff[p], qoff[p + 1])
        sub = wl.DecodeWorkload("page", [pg], w.Hq, w.Hkv, w.d, w.value_scale)
        vals = wl.DecodeValues([hv["prefix_k"]], [hv["prefix_v"]], hv["own_k"], hv["own_v"], q_host[rows],
                               kn_host[rows], vn_host[rows])
        O, L = ta.branch_decode(sub, vals, tree=tree)
        check(o[rows], lse[rows], O, L, "bf16", f"page {p}")
    del d
    torch.cuda.empty_cache()


def test_serving_decode_sampled_pages(harness):
    """512 pages, about 17.6 k branches, a 48 GB pool: 6 sampled pages."""
    w = wl.serving_decode(0)
    _decode_sampled(harness, w, False, [0, 101, 257, 384, 450, 511])


def test_spec_verify_sampled_pages(harness):
    """64 pages with draft trees of up to 16 nodes: 6 sampled pages."""
    w = wl.spec_verify(0)
    _decode_sampled(harness, w, True, [0, 9, 20, 33, 47, 63])


def test_packed_forward_sampled_rows(harness):
    """8 packed sequences of 16384 tokens; sampled rows of 4 pages."""
    import torch
    fw = wl.packed_sequences(0)
    f = harness.Forward(fw, seed=0)
    o, lse = f.run()
    torch.cuda.synchronize()
    padoc.device_status()
    starts = np.cumsum([0] + [p.n_tokens for p in fw.pages])
    rng = np.random.default_rng(0)
    for pi in [0, 3, len(fw.pages) // 2, len(fw.pages) - 1]:
        a, b = int(starts[pi]), int(starts[pi + 1])
        page = [fw.pages[pi]]
        q = f.q[a:b].float().cpu().numpy()
        k = f.k[a:b].float().cpu().numpy()
        v = f.v[a:b].float().cpu().numpy()
        n = b - a
        rows = sorted(set(rng.choice(n, min(n, 96), replace=False).tolist()) | {0, n - 1})
        O, L = ta.tree_forward(q, k, v, page, positions=rows)
        og = o[a:b].float().cpu().numpy()[rows]
        lg = lse[:, a:b].cpu().numpy()[:, rows]
        check(og, lg, O[rows], L[:, rows], "bf16", f"packed page {pi}")


def test_packed_forward_whole_page(harness, tmp_path):
    """8 packed sequences of 16384 tokens in one launch, checked on every row
    of one whole page (the smallest with a prefix, layout and content), so
    every region boundary of the page, where a causal own segment starts,
    and every tile edge is covered.  The oracle runs in a spawned pool."""
    import torch
    from parity import pooled_forward
    fw = wl.packed_sequences(0)
    f = harness.Forward(fw, seed=0)
    o, lse = f.run()
    torch.cuda.synchronize()
    padoc.device_status()
    starts = np.cumsum([0] + [p.n_tokens for p in fw.pages])
    cand = [i for i, pg in enumerate(fw.pages) if sum(pg.layout_len) > 0 and sum(pg.content_len) > 0]
    pi = min(cand, key=lambda i: fw.pages[i].n_tokens)
    a, b = int(starts[pi]), int(starts[pi + 1])
    host = [x[a:b].float().cpu().numpy() for x in (f.q, f.k, f.v)]
    path = str(tmp_path / "page.npz")
    np.savez(path, q=host[0], k=host[1], v=host[2])
    O, L = pooled_forward(path, [fw.pages[pi]], b - a, fw.Hq, fw.d)
    check(o[a:b].float().cpu().numpy(), lse[:, a:b].cpu().numpy(), O, L, "bf16", f"packed page {pi}, all rows")

