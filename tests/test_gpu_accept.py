"""Accept step and commit on the GPU against the oracle.

The accept outputs (accepted length, path, free token) are integers decided
from bf16 logits in float32 on both sides, so they must agree bit for bit.
The commit moves bytes, so the pool must hold exactly the committed rows."""
import numpy as np
import pytest

from oracle import accept as acc
from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu_accept(logits, tokens, parents, q_offsets, tau, max_nodes=16, offset=0):
    """Runs padoc_verify_accept; `offset` shifts the logits base by that many
    bf16 elements (an unaligned start takes the scalar load path)."""
    import torch
    nq, V = logits.shape
    flat = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).to(torch.bfloat16).reshape(-1)
    buf = torch.zeros(nq * V + offset + 8, dtype=torch.bfloat16, device="cuda")
    buf[offset:offset + nq * V] = flat.cuda()
    lg = buf[offset:]
    B = len(q_offsets) - 1
    n_acc = torch.full((B,), 77, dtype=torch.int32, device="cuda")
    path = torch.full((B, 16), 77, dtype=torch.int32, device="cuda")
    free = torch.full((B,), 77, dtype=torch.int32, device="cuda")
    padoc.verify_accept(lg, nq, V, _dev(np.asarray(tokens, np.int32)), _dev(np.asarray(parents, np.int32)),
                        _dev(np.asarray(q_offsets, np.int32)), B, max_nodes, tau, n_acc, path, free)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), path.cpu().numpy(), free.cpu().numpy()


def _same(got, want, what):
    for g, e, name in zip(got, want, ("n_acc", "path", "free_token")):
        bad = np.nonzero(np.asarray(g).reshape(len(g), -1) != np.asarray(e).reshape(len(e), -1))[0]
        assert len(bad) == 0, f"{what}: {name} differs at branches {bad[:8].tolist()}: {g[bad[:4]]} vs {e[bad[:4]]}"


def _trees(seed, n):
    rng = np.random.default_rng(seed)
    return [wl.draft_tree(rng) for _ in range(n)]


@pytest.mark.parametrize("V", [1000, 4096, 32776])
@pytest.mark.parametrize("tau", [0.75, 1.0, 0.5])
def test_accept_matches_oracle(padoc_lib, V, tau):
    trees = _trees(V, 40)
    inp = wl.accept_inputs(V + int(tau * 100), trees, V)
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, tau)
    got = _gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, tau)
    _same(got, want, f"V={V} tau={tau}")
    assert want[0].max() >= 2  # the recipe yields multi-token accepts


@pytest.mark.parametrize("V", [64, 1000])
@pytest.mark.parametrize("tau", [1.0, 0.75])
def test_accept_ties_go_to_lowest_index(padoc_lib, V, tau):
    """Small-integer logits: equal scores everywhere (u_hat and children)."""
    trees = _trees(7 + V, 60)
    inp = wl.accept_inputs(3 + V, trees, V, ties=True)
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, tau)
    got = _gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, tau)
    _same(got, want, f"ties V={V} tau={tau}")


def test_accept_chains_and_single_nodes(padoc_lib):
    """Chains of 1..16 nodes (the HPD-Parsing drafted window) and
    single-node branches under max_nodes = 1 (plain decode)."""
    chains = [[-1] + list(range(n - 1)) for n in range(1, 17)] * 3
    inp = wl.accept_inputs(11, chains, 2048, p_agree=0.85)
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 1.0)
    _same(_gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 1.0), want, "chains")
    single = [[-1]] * 37
    inp = wl.accept_inputs(12, single, 3000)
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75)
    got = _gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75, max_nodes=1)
    _same(got, want, "single nodes")
    assert (got[0] == 0).all()


@pytest.mark.parametrize("offset", [1, 3])
def test_accept_unaligned_logits(padoc_lib, offset):
    trees = _trees(21, 12)
    inp = wl.accept_inputs(21, trees, 4096)
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75)
    _same(_gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75, offset=offset), want, "unaligned")


def test_accept_special_rows(padoc_lib):
    """Maximum in the last column, a constant row, and -inf scores (a child
    at -inf against a -inf maximum gives NaN and is rejected on both sides)."""
    V = 1024
    trees = [[-1, 0, 0, 1], [-1, 0, 1], [-1, 0]]
    inp = wl.accept_inputs(5, trees, V)
    L = inp.logits
    L[0, :] = -1.0
    L[0, V - 1] = 9.0
    L[0, inp.tokens[1]] = 9.0  # node 1 ties the row maximum: accepted, u_hat the lower index
    L[4, :] = 0.25          # branch 1, node 0: constant row, argmax 0
    L[5, :] = -np.inf       # branch 1, node 1: -inf everywhere
    L[7, :] = -np.inf       # branch 2, node 0
    with np.errstate(invalid="ignore"):
        want = acc.accept_batch(L, inp.tokens, inp.parents, inp.q_offsets, 0.75)
    _same(_gpu_accept(L, inp.tokens, inp.parents, inp.q_offsets, 0.75), want, "special rows")


def test_accept_invalid_branches_are_flagged(padoc_lib):
    V = 512
    trees = [[-1, 0, 1], [-1, 0, 0], [-1, 0, 1, 2], [-1, 0], [-1, 0, 0, 1, 1]]
    inp = wl.accept_inputs(9, trees, V)
    par, tok = inp.parents.copy(), inp.tokens.copy()
    qo = inp.q_offsets
    par[qo[1] + 2] = 2      # branch 1: a node that is its own parent
    tok[qo[2] + 3] = V      # branch 2: token outside the vocabulary
    par[qo[3]] = 0          # branch 3: node 0 with a parent
    want = acc.accept_batch(inp.logits, inp.tokens, inp.parents, qo, 0.75)
    n_acc, path, free = _gpu_accept(inp.logits, tok, par, qo, 0.75, max_nodes=4)
    for b in (1, 2, 3, 4):  # branch 4 has 5 nodes > max_nodes = 4
        assert n_acc[b] == -1 and free[b] == -1 and (path[b] == -1).all(), b
    assert n_acc[0] == want[0][0] and (path[0] == want[1][0]).all() and free[0] == want[2][0]
    # empty branch (q_offsets repeat) and a branch whose rows leave [0, nq)
    qo2 = np.array([0, 3, 3, 5], np.int32)
    n_acc, path, free = _gpu_accept(inp.logits[:4], inp.tokens[:4], inp.parents[:4], qo2, 0.75)
    assert n_acc[1] == -1 and n_acc[2] == -1
    assert n_acc[0] == want[0][0] and free[0] == want[2][0]


def test_accept_full_vocab_verify_batch(padoc_lib):
    """The 64-page verify batch (about 13k draft nodes) against the full
    151,936-token vocabulary, logits drawn on the GPU; branches sampled for
    the oracle, and every output checked for validity."""
    import torch
    w = wl.spec_verify(0)
    trees = [t for pg in w.pages for t in pg.parents]
    inp = wl.DeviceAcceptInputs(3, trees, wl.VOCAB, "cuda")
    B = len(trees)
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty(B, 16, dtype=torch.int32, device="cuda")
    free = torch.empty(B, dtype=torch.int32, device="cuda")
    padoc.verify_accept(inp.logits, inp.nq, inp.vocab, _dev(inp.tokens), _dev(inp.parents), _dev(inp.q_offsets),
                        B, 16, 0.75, n_acc, path, free)
    torch.cuda.synchronize()
    n_acc, path, free = n_acc.cpu().numpy(), path.cpu().numpy(), free.cpu().numpy()
    assert (n_acc >= 0).all() and (free >= 0).all() and (free < wl.VOCAB).all()
    rng = np.random.default_rng(0)
    qo = inp.q_offsets
    for b in sorted(rng.choice(B, 48, replace=False).tolist()) + [0, B - 1]:
        rows = inp.host_rows(range(qo[b], qo[b + 1]))
        p, f = acc.accept_tree(rows, inp.tokens[qo[b]:qo[b + 1]], inp.parents[qo[b]:qo[b + 1]], 0.75)
        assert n_acc[b] == len(p) and path[b, :len(p)].tolist() == p and (path[b, len(p):] == -1).all(), b
        assert free[b] == f, b
    assert n_acc.max() >= 3  # the recipe yields multi-token accepts


# ---------------------------------------------------------------------------- commit


def test_commit_writes_exact_rows(padoc_lib):
    """Commit rows into forked branches (fork lengths off block boundaries,
    commits crossing blocks); every slot of every sequence is read back, and
    the parent's shared blocks stay untouched."""
    import torch
    Hkv, d, nb = 2, 128, 64
    kp = torch.zeros(nb, Hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = padoc.KVPool(kp, vp, nb, Hkv, d, max_seqs=16, max_blocks_per_seq=12)
    pool.sync()
    rnd = lambda s, n: torch.from_numpy(wl.round_bf16(wl.normal_f32(s, (n, Hkv, d)))).to(torch.bfloat16).cuda()
    P = 37
    pk, pv = rnd(1, P), rnd(2, P)
    page = pool.alloc(P)
    pool.append(page, pk, pv, P)
    own_n = [0, 5, 16, 30]
    forks, own_k, own_v = [], [], []
    for i, n in enumerate(own_n):
        c = pool.fork(page, P - 3 * i)
        k, v = rnd(10 + i, max(n, 1)), rnd(20 + i, max(n, 1))
        if n:
            pool.append(c, k, v, n)
        forks.append(c)
        own_k.append(k[:n])
        own_v.append(v[:n])
    nsrc = 40
    kn, vn = rnd(50, nsrc), rnd(51, nsrc)
    rng = np.random.default_rng(3)
    counts = [17, 0, 3, 12]
    rows = [rng.choice(nsrc, c, replace=False).astype(np.int32) for c in counts]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = torch.empty(16 * int(offs[-1]), dtype=torch.uint8, device="cuda")
    shared_before = [kp[int(b)].clone() for b in pool.seq_blocks(page)]
    pool.commit(forks, offs, np.concatenate(rows), nsrc, kn, vn, ws, ws.numel())
    torch.cuda.synchronize()
    for i, c in enumerate(forks):
        info = pool.seq_info(c)
        fl = info["fork_len"]
        assert info["length"] == fl + own_n[i] + counts[i]
        blocks = pool.seq_blocks(c)
        nsh = (fl + 15) // 16
        want_k = torch.cat([own_k[i], kn[torch.from_numpy(rows[i]).long().cuda()]])
        want_v = torch.cat([own_v[i], vn[torch.from_numpy(rows[i]).long().cuda()]])
        for t in range(own_n[i] + counts[i]):
            blk = int(blocks[nsh + t // 16])
            assert torch.equal(kp[blk, :, t % 16], want_k[t]), (i, t)
            assert torch.equal(vp[blk, :, t % 16], want_v[t]), (i, t)
    for b, before in zip(pool.seq_blocks(page), shared_before):
        assert torch.equal(kp[int(b)], before)


def _single_root_workload(seed, n_pages=3):
    rng = np.random.default_rng(seed)
    pages = []
    for _ in range(n_pages):
        P = int(rng.integers(20, 300))
        N = int(rng.integers(1, 5))
        own = rng.integers(0, 60, N).tolist()
        trees = [wl.draft_tree(rng) for _ in range(N)]
        pages.append(wl.DecodePage(P, [P] * N, own, [len(t) for t in trees], trees))
    return wl.DecodeWorkload("verify_then_decode", pages, 4, 2, 128, 1.0)


@pytest.mark.parametrize("seed", [0, 1])
def test_verify_accept_commit_next_step(padoc_lib, seed):
    """One full speculative round: verify the draft trees, accept on
    synthetic logits, commit the anchor and accepted nodes, then decode the
    next anchor over the grown cache; the oracle sees the committed rows as
    ordinary own-suffix tokens."""
    import torch
    from tree_structured_shared_gb300 import harness
    w = _single_root_workload(seed)
    vals = wl.decode_values(w, seed)
    dec = harness.Decode(w, vals, slack_blocks=2 * w.n_branches + 8)
    o, lse = dec.run()
    torch.cuda.synchronize()
    O, L = ta.branch_decode(w, vals)
    check(o.float().cpu().numpy()[: w.n_queries], lse.cpu().numpy()[: w.n_queries], O, L, "bf16", "verify")

    trees = [t for pg in w.pages for t in pg.parents]
    inp = wl.accept_inputs(seed, trees, 640, p_agree=0.8)
    n_acc, path, free = _gpu_accept(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75)
    _same((n_acc, path, free), acc.accept_batch(inp.logits, inp.tokens, inp.parents, inp.q_offsets, 0.75), "accept")

    qo = inp.q_offsets
    rows = [np.concatenate([[qo[b]], qo[b] + path[b, :n_acc[b]]]).astype(np.int32) for b in range(len(trees))]
    offs = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ws = torch.empty(16 * int(offs[-1]), dtype=torch.uint8, device="cuda")
    dec.pool.commit(dec.branch_seq, offs, np.concatenate(rows), dec.nq, dec.k_new, dec.v_new, ws, ws.numel())

    B = len(trees)
    bo = [0]
    for pg in w.pages:
        bo.append(bo[-1] + len(pg.own_len))
    batch2 = padoc.Batch(dec.page_seq, bo, dec.branch_seq, list(range(B + 1)))
    s2 = 1000 + seed
    q2 = wl.round_bf16(wl.normal_f32(s2, (B, w.Hq, w.d)))
    k2 = wl.round_bf16(wl.normal_f32(s2 + 1, (B, w.Hkv, w.d)))
    v2 = wl.round_bf16(wl.normal_f32(s2 + 2, (B, w.Hkv, w.d)))
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    wsb = padoc.branch_decode_ws_size(dec.pool, batch2, w.Hq)
    ws2 = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    o2 = torch.empty(B, w.Hq, w.d, dtype=torch.bfloat16, device="cuda")
    l2 = torch.empty(B, w.Hq, dtype=torch.float32, device="cuda")
    padoc.branch_decode(dec.pool, batch2, w.Hq, bf(q2), bf(k2), bf(v2), None, o2, l2, ws2, wsb)
    torch.cuda.synchronize()

    pages2, own_k, own_v = [], [], []
    b = 0
    for pg in w.pages:
        grown = []
        for j in range(len(pg.own_len)):
            own_k.append(np.concatenate([vals.own_k[b], vals.k_new[rows[b]]]))
            own_v.append(np.concatenate([vals.own_v[b], vals.v_new[rows[b]]]))
            grown.append(pg.own_len[j] + len(rows[b]))
            b += 1
        n = len(pg.own_len)
        pages2.append(wl.DecodePage(pg.prefix_len, pg.branch_prefix_len, grown, [1] * n, [[-1]] * n))
    w2 = wl.DecodeWorkload("next_step", pages2, w.Hq, w.Hkv, w.d, 1.0)
    vals2 = wl.DecodeValues(vals.prefix_k, vals.prefix_v, own_k, own_v, q2, k2, v2)
    O2, L2 = ta.branch_decode(w2, vals2, tree=False)
    check(o2.float().cpu().numpy(), l2.cpu().numpy(), O2, L2, "bf16", "next step after commit")
