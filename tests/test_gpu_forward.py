"""Tree-varlen forward on the GPU against the float64 oracle."""
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


def _run(harness, w, seed=0, order=padoc.PACK_CANONICAL, positions=None):
    q, k, v = wl.tree_qkv(w, seed)
    f = harness.Forward(w, q, k, v, order=order)
    o, lse = f.run()
    import torch
    torch.cuda.synchronize()
    padoc.device_status()
    O, L = ta.tree_forward(q, k, v, w.pages, order, positions=positions)
    og = o.float().cpu().numpy()[: w.n_tokens]
    lg = lse.cpu().numpy()[:, : w.n_tokens]
    if positions is not None:
        pos = np.asarray(positions)
        return og[pos], lg[:, pos], O[pos], L[:, pos]
    return og, lg, O, L


def test_tiny_fp32_page(harness):
    w = wl.tiny_fp32_page(0)
    og, lg, O, L = _run(harness, w)
    check(og, lg, O, L, "f32", "tiny fp32 page")


@pytest.mark.parametrize("seed", [0, 1])
def test_qwen_page_bf16_every_row(harness, seed, tmp_path):
    """The Qwen-shaped page (X = 2048, 24 regions, lognormal content) on
    every row: all tile edges, every region's first layout and content token
    (where a causal own segment starts) and every ragged tail.  The oracle
    runs in a pool of spawned processes."""
    from parity import pooled_forward
    w = wl.qwen_page(seed)
    q, k, v = wl.tree_qkv(w, seed)
    f = harness.Forward(w, q, k, v)
    o, lse = f.run()
    import torch
    torch.cuda.synchronize()
    padoc.device_status()
    path = str(tmp_path / "qkv.npz")
    np.savez(path, q=q, k=k, v=v)
    O, L = pooled_forward(path, w.pages, w.n_tokens, w.Hq, w.d)
    check(o.float().cpu().numpy()[: w.n_tokens], lse.cpu().numpy()[:, : w.n_tokens], O, L, "bf16",
          f"qwen page seed {seed}, all {w.n_tokens} rows")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("order", [padoc.PACK_CANONICAL, padoc.PACK_DOCUMENT])
def test_random_pages_bf16_full(harness, G, order):
    """Several pages, ragged regions (empty ones included), several tiles."""
    w = wl.random_pages(10 + G, n_pages=3, max_prefix=300, max_regions=6, max_layout=20, max_content=150,
                        Hq=2 * G, Hkv=2, d=128, dtype="bf16")
    og, lg, O, L = _run(harness, w, seed=G, order=order)
    check(og, lg, O, L, "bf16", f"random pages G={G} order={order}")


def test_one_region_page_is_causal_attention(harness):
    w = wl.TreeWorkload("causal", [wl.Page(300, [20], [200])], 4, 2, 128, "bf16", 1.0, [0])
    og, lg, O, L = _run(harness, w, seed=3)
    check(og, lg, O, L, "bf16", "one region")


def test_isolation_bit_exact(harness):
    """Perturbing branch Y_j changes no other token's output bit."""
    import torch
    w = wl.random_pages(5, n_pages=1, max_prefix=200, max_regions=5, max_layout=10, max_content=100,
                        allow_empty=False, Hq=4, Hkv=2, d=128, dtype="bf16")
    q, k, v = wl.tree_qkv(w, 1)
    f1 = harness.Forward(w, q, k, v)
    o1, l1 = [x.clone() for x in f1.run()]
    ident, pos = ta.packed_layout(w.pages)
    yj = [pos[(0, ta.Y_KIND, 2, i)] for i in range(w.pages[0].content_len[2])]
    k2, v2 = k.copy(), v.copy()
    k2[yj] = wl.round_bf16(k2[yj] + 1.0)
    v2[yj] = wl.round_bf16(v2[yj] * -2.0)
    f2 = harness.Forward(w, q, k2, v2)
    o2, l2 = f2.run()
    torch.cuda.synchronize()
    others = [t for t in range(w.n_tokens) if t not in set(yj)]
    assert torch.equal(o1[others], o2[others])
    assert torch.equal(l1[:, others], l2[:, others])
    assert not torch.equal(o1[yj], o2[yj])


def test_empty_and_tiny(harness):
    import torch
    w = wl.TreeWorkload("e", [], 4, 2, 128, "bf16", 1.0, [])
    f = harness.Forward(w, np.zeros((0, 4, 128), np.float32), np.zeros((0, 2, 128), np.float32),
                        np.zeros((0, 2, 128), np.float32))
    f.run()
    torch.cuda.synchronize()
    w = wl.TreeWorkload("one", [wl.Page(1, [], [])], 4, 2, 128, "bf16", 1.0, [0])
    og, lg, O, L = _run(harness, w)
    check(og, lg, O, L, "bf16", "single token")


def test_unsupported_shapes_rejected(harness):
    w = wl.TreeWorkload("x", [wl.Page(8, [], [])], 6, 2, 128, "bf16", 1.0, [0])  # group 3
    with pytest.raises(padoc.PadocError):
        harness.Forward(w)


def test_repeat_runs_bit_identical(harness):
    """Many units of many key tiles, run repeatedly: any ordering race in the
    pipeline shows up as a difference between runs."""
    import torch
    w = wl.packed_sequences(3, n_seq=1, seq_tokens=16384)
    f = harness.Forward(w, seed=3)
    o0, l0 = [x.clone() for x in f.run()]
    for _ in range(4):
        o, l = f.run()
        torch.cuda.synchronize()
        assert torch.equal(o, o0) and torch.equal(l, l0)
    padoc.device_status()


def test_output_16_byte_aligned(harness):
    """An output tensor that is 16- but not 32-byte aligned (the ABI's
    promise): the epilogue stores each row in 16-byte pieces instead of
    32-byte ones.  Random bf16 pages against the oracle."""
    import torch
    w = wl.random_pages(31, n_pages=2, max_prefix=300, max_regions=5, max_layout=20, max_content=150,
                        Hq=4, Hkv=2, d=128, dtype="bf16")
    q, k, v = wl.tree_qkv(w, 31)
    f = harness.Forward(w, q, k, v)
    buf = torch.empty(f.o.numel() + 8, dtype=f.o.dtype, device=f.o.device)
    f.o = buf[8:].view(f.o.shape)
    assert f.o.data_ptr() % 32 == 16
    o, lse = f.run()
    torch.cuda.synchronize()
    padoc.device_status()
    O, L = ta.tree_forward(q, k, v, w.pages)
    check(o.float().cpu().numpy()[: w.n_tokens], lse.cpu().numpy()[:, : w.n_tokens], O, L, "bf16",
          "16-byte aligned output")
