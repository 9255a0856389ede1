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
