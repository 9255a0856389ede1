"""The allocation-free decode entry point (padoc_branch_decode_noalloc).

It exists for callers that may not allocate device memory themselves, for
example code running inside a host runtime that owns all GPU memory through
its own arena, so they cannot hand over a workspace.  The entry point takes
its workspace from a fixed device array inside the library.  These tests
call it through the C ABI and compare it with padoc_branch_decode, which
uses a caller-provided workspace, on two calls in a row (the second call
finds the array holding the first call's contents).
"""
import numpy as np
import pytest

from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def harness(padoc_lib):
    from tree_structured_shared_gb300 import harness as h
    return h


def _compare_two_calls(harness, w, vals, tree):
    import torch
    d = harness.Decode(w, vals, tree=tree)
    o_ref, l_ref = [x.clone() for x in d.run()]
    torch.cuda.synchronize()
    assert d.ws_bytes <= padoc.NOALLOC_SCRATCH_BYTES
    nq = w.n_queries
    for call in range(2):
        o = torch.full_like(d.o, float("nan"))
        lse = torch.full_like(d.lse, float("nan"))
        padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
        torch.cuda.synchronize()
        padoc.device_status()
        check(o.float().cpu().numpy()[:nq], lse.cpu().numpy()[:nq], o_ref.float().cpu().numpy()[:nq],
              l_ref.cpu().numpy()[:nq], "bf16", f"no-alloc call {call}")


def test_noalloc_matches_workspace_entry_point_verify(harness):
    w = wl.small_decode(5, n_pages=4, max_prefix=600, max_branches=6, max_own=250, Hq=4, Hkv=2)
    _compare_two_calls(harness, w, wl.decode_values(w, 5), tree=True)


def test_noalloc_matches_workspace_entry_point_branch_decode(harness):
    w = wl.branch_decode(2)  # 16 pages, prefix 4809, 8-40 branches, one query each
    _compare_two_calls(harness, w, None, tree=False)


def test_noalloc_rejects_oversized_step(harness):
    """A step whose workspace exceeds the fixed array is refused up front."""
    import torch
    n_pages, n_br, ql = 40, 60, 16
    k = torch.zeros(n_pages + 8, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    pool = padoc.KVPool(k, v, n_pages + 8, Hkv=2, d=128, max_seqs=n_pages * (n_br + 1) + 8, max_blocks_per_seq=4)
    pool.sync()
    one = torch.zeros(16, 2, 128, dtype=torch.bfloat16, device="cuda")
    page_seq, br, boff, qoff = [], [], [0], [0]
    for _ in range(n_pages):
        s = pool.alloc(16)
        pool.append(s, one, one, 16)
        page_seq.append(s)
        for _ in range(n_br):
            br.append(pool.fork(s, 16))
            qoff.append(qoff[-1] + ql)
        boff.append(len(br))
    batch = padoc.Batch(page_seq, boff, br, qoff)
    assert padoc.branch_decode_ws_size(pool, batch, 16) > padoc.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(padoc.PadocError) as e:
        padoc.branch_decode_noalloc(pool, batch, 16, dummy, dummy, dummy, None, dummy, dummy)
    assert e.value.code == padoc.ERR_INVALID and "scratch" in str(e.value)
    torch.cuda.synchronize()


def test_noalloc_requires_set_up_pool(harness):
    """Without padoc_kv_pool_sync at set-up the pool has no device table, and
    creating one would allocate: the call is refused."""
    import torch
    k = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    pool = padoc.KVPool(k, torch.zeros_like(k), 4, Hkv=2, d=128, max_seqs=4, max_blocks_per_seq=2)
    s = pool.alloc(0)
    c = pool.fork(s, 0)
    batch = padoc.Batch([s], [0, 1], [c], [0, 1])
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 4, dtype=torch.float32, device="cuda")
    with pytest.raises(padoc.PadocError) as e:
        padoc.branch_decode_noalloc(pool, batch, 4, q, kv, kv, None, o, lse)
    assert e.value.code == padoc.ERR_INVALID and "padoc_kv_pool_sync" in str(e.value)
