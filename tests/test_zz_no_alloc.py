"""The allocation-free decode entry point (padoc_branch_decode_noalloc).

It exists for callers that may not allocate device memory themselves, for
example code running inside a host runtime that owns all GPU memory through
its own arena, so they cannot hand over a workspace.  The entry point takes
its workspace from a fixed device array inside the library.  These tests
call it through the C ABI and require it to reproduce padoc_branch_decode,
which uses a caller-provided workspace, bit for bit on two calls in a row
(the second call finds the array holding the first call's contents); one
case is also checked against the float64 oracle.  They also check that a
call leaves the device's free memory unchanged, and the refusals: a step
too large for the array, a pool without its device table, a pool whose
table lives on another device.
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
    """Two calls in a row must reproduce padoc_branch_decode bit for bit: the
    kernels and the plan are the same, only the workspace address differs.
    Returns the no-alloc call's outputs (the queries' rows)."""
    import torch
    d = harness.Decode(w, vals, tree=tree)
    o_ref, l_ref = [x.clone() for x in d.run()]
    torch.cuda.synchronize()
    assert d.ws_bytes <= padoc.NOALLOC_SCRATCH_BYTES
    nq = w.n_queries
    out = None
    for call in range(2):
        o = torch.full_like(d.o, float("nan"))
        lse = torch.full_like(d.lse, float("nan"))
        padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
        torch.cuda.synchronize()
        padoc.device_status()
        assert torch.equal(o[:nq], o_ref[:nq]), f"no-alloc call {call}: O differs from padoc_branch_decode"
        assert torch.equal(lse[:nq], l_ref[:nq]), f"no-alloc call {call}: LSE differs from padoc_branch_decode"
        out = (o[:nq].float().cpu().numpy(), lse[:nq].cpu().numpy())
    return d, out


def test_noalloc_matches_workspace_entry_point_verify(harness):
    """Draft trees on ragged pages: bit-identical to the workspace entry
    point, and within the bf16 tolerances of the float64 oracle."""
    from oracle import tree_attention as ta
    w = wl.small_decode(5, n_pages=4, max_prefix=600, max_branches=6, max_own=250, Hq=4, Hkv=2)
    vals = wl.decode_values(w, 5)
    _, (o, lse) = _compare_two_calls(harness, w, vals, tree=True)
    O, L = ta.branch_decode(w, vals, tree=True)
    check(o, lse, O, L, "bf16", "no-alloc verify against the oracle")


def test_noalloc_matches_workspace_entry_point_branch_decode(harness):
    w = wl.branch_decode(2)  # 16 pages, prefix 4809, 8-40 branches, one query each
    _compare_two_calls(harness, w, None, tree=False)


def test_noalloc_call_takes_no_device_memory(harness):
    """After a first call (which may load the module and so reserve the
    array), a call leaves the device's free memory exactly as it was."""
    import torch
    w = wl.small_decode(6, n_pages=3, max_prefix=500, max_branches=5, max_own=200, Hq=4, Hkv=2)
    d = harness.Decode(w, wl.decode_values(w, 6), tree=True)
    o, lse = torch.empty_like(d.o), torch.empty_like(d.lse)
    padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    padoc.device_status()
    assert free1 == free0, (free0, free1)


def test_noalloc_empty_batch(harness):
    """A step with no branches returns at once and touches nothing."""
    import torch
    k = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    pool = padoc.KVPool(k, torch.zeros_like(k), 4, Hkv=2, d=128, max_seqs=4, max_blocks_per_seq=2)
    pool.sync()
    batch = padoc.Batch([], [0], [], [0])
    o = torch.full((1, 4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 4), 7.0, dtype=torch.float32, device="cuda")
    padoc.branch_decode_noalloc(pool, batch, 4, o, o, o, None, o, lse)
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())


def test_noalloc_rejects_other_device(harness):
    """The scratch address belongs to the current device, so a pool whose
    table lives on another device is refused before any launch; the same
    call succeeds once the pool's device is current again."""
    import torch
    w = wl.small_decode(7, n_pages=2, max_prefix=300, max_branches=3, max_own=80, Hq=4, Hkv=2)
    d = harness.Decode(w, wl.decode_values(w, 7), tree=True)
    dev = d.pool.device()
    assert dev == torch.cuda.current_device()
    o, lse = torch.empty_like(d.o), torch.empty_like(d.lse)
    d.pool.debug_rehome(dev + 1)
    try:
        with pytest.raises(padoc.PadocError) as e:
            padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
        assert e.value.code == padoc.ERR_INVALID and "device" in str(e.value)
        with pytest.raises(padoc.PadocError):
            d.run()  # the workspace entry point checks the same before its upload
    finally:
        d.pool.debug_rehome(dev)
    padoc.branch_decode_noalloc(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, d.tree_bits, o, lse)
    torch.cuda.synchronize()
    padoc.device_status()


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
