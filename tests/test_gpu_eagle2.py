"""GPU parity of the EAGLE-2 tree budget with the oracle.

* spec_topk: tokens bit-exact (ties to the lower index), probabilities within
  1e-5 relative of the fp64 oracle; both element types, masked entries, exact
  ties, unaligned rows (plain loads), k from 1 to 32.
* The whole budget loop: both sides grow their own trees from the same
  stand-in draft model (a node's row depends only on its token path), step by
  step, then rerank.  Trees must be identical except for sequences where the
  oracle flags a selection boundary within 1e-5 (fp32 values on the GPU,
  fp64 in the oracle); those may differ, at most one per test.
* Errors: a frontier id outside the tree, a malformed tree for the rerank.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import record_parity
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import (EAGLE2_WORKLOADS, Eagle2Workload, draft_rows, node_key,
                                                 root_key)

pytestmark = pytest.mark.gpu


def _rows(R, V, dtype, seed, ties=True, masked=True):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = torch.randn((R, V), generator=g, device="cuda") * 3
    if ties:
        z[:, ::3] = torch.round(z[:, ::3])   # exact ties, among them -0.0 and +0.0
    if masked and V > 8:
        z[0, : V // 2] = float("-inf")
    return z.to(torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()


TOPK = [(3, 7, 3, "f32", 1.0), (16, 1000, 10, "bf16", 1.0), (9, 4097, 16, "f32", 0.7), (40, 32000, 8, "bf16", 1.3),
        (64, 128256, 10, "bf16", 1.0), (5, 128256, 32, "f32", 1.0), (300, 5000, 1, "bf16", 2.0),
        (7, 50, 32, "f32", 1.0)]


@pytest.mark.parametrize("R,V,k,dtype,T", TOPK, ids=[f"R{c[0]}V{c[1]}k{c[2]}{c[3]}T{c[4]}" for c in TOPK])
def test_topk_parity(R, V, k, dtype, T):
    z = _rows(R, V, dtype, seed=R * 7 + V)
    tok, prob = binding.spec_topk(z, k, T)
    assert binding.spec_get_status() == 0
    rt, rp = oracle.topk_prob(z.cpu(), k, T)
    assert np.array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=1e-5, atol=1e-30)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_topk_cluster_sizes(G, monkeypatch):
    """Rows split over G CTAs of a cluster merge to the same answer
    (SPEC_TOPK_CLUSTER overrides the choice)."""
    monkeypatch.setenv("SPEC_TOPK_CLUSTER", str(G))
    for R, V, k, dtype in ((5, 128256, 10, "bf16"), (3, 40000, 32, "f32"), (4, 1003, 8, "bf16")):
        z = _rows(R, V, dtype, seed=G * 100 + V)
        tok, prob = binding.spec_topk(z, k, 1.0)
        rt, rp = oracle.topk_prob(z.cpu(), k, 1.0)
        assert np.array_equal(tok.cpu().numpy(), rt)
        np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=1e-5, atol=1e-30)


@pytest.mark.parametrize("dtype,spread", [("bf16", 3), ("bf16", 9), ("f32", 5)])
def test_topk_best_elements_in_one_thread(dtype, spread, monkeypatch):
    """A thread reads every 512th 16-byte vector of its CTA's slice.  Put the
    row's best elements in vectors 512 apart (one thread's) and that
    thread's other vectors reach the threshold too, so it re-reads all of
    them instead of offering its best vector alone; the results must not
    change."""
    monkeypatch.setenv("SPEC_TOPK_CLUSTER", "1")  # one CTA per row: the slice starts at 0
    R, V, k = 6, 128256, 8
    z = _rows(R, V, dtype, seed=spread, ties=False, masked=False).float()
    ve = 4 if dtype == "f32" else 8
    for r in range(R):
        v0 = 17 + 29 * r
        for j in range(spread):
            z[r, (v0 + 512 * j) * ve + (j % ve)] = 60.0 - j
    z = z.to(torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()
    tok, prob = binding.spec_topk(z, k, 1.0)
    assert binding.spec_get_status() == 0
    rt, rp = oracle.topk_prob(z.cpu(), k, 1.0)
    assert np.array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=1e-5, atol=1e-30)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_topk_flat_and_masked_rows(dtype):
    """Rows where thousands of entries reach the threshold (all equal; or all
    -inf but three) take the lockstep-admission path; ties go to the lowest
    indices."""
    V, k = 50000, 8
    z = torch.zeros((3, V), device="cuda")
    z[1] = float("-inf")
    z[1, [7, 20000, 49999]] = torch.tensor([1.0, 3.0, 2.0], device="cuda")
    z[2, ::2] = 1.5                       # half the row ties at the maximum
    z = z.to(torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()
    tok, prob = binding.spec_topk(z, k, 1.0)
    assert binding.spec_get_status() == 0
    rt, rp = oracle.topk_prob(z.cpu(), k, 1.0)
    assert np.array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=1e-5, atol=1e-30)
    assert tok[0].tolist() == list(range(k)) and tok[2].tolist() == list(range(0, 2 * k, 2))


def test_topk_unaligned_rows():
    base = _rows(1, 1001 * 6 + 1, "bf16", seed=3, masked=False).reshape(-1)
    z = base[1:].view(6, 1001)                  # odd V, data pointer 2 bytes off: plain loads
    tok, prob = binding.spec_topk(z, 12, 1.0)
    rt, rp = oracle.topk_prob(z.cpu(), 12, 1.0)
    assert np.array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=1e-5)


def test_bad_frontier_and_malformed_tree():
    B, V, k = 2, 100, 4
    z = _rows(B * 2, V, "f32", seed=1).view(B, 2, V)
    tok = torch.zeros((B, 20), dtype=torch.int32, device="cuda")
    val = torch.ones((B, 20), dtype=torch.float32, device="cuda")
    par = torch.full((B, 20), -1, dtype=torch.int32, device="cuda")
    frontier = torch.tensor([[0, 0], [0, 5]], dtype=torch.int32, device="cuda")   # 5 is not yet a node
    nxt = binding.spec_eagle2_expand(z, frontier, tok, val, par, k, 1, 3)
    assert binding.spec_get_status() == 7
    assert nxt[1].tolist() == [-1, -1, -1] and min(nxt[0].tolist()) >= 1
    bad = torch.tensor([[-1, 0, 2, 1]], dtype=torch.int32, device="cuda")           # parent after its child
    out = binding.spec_eagle2_rerank(torch.ones((1, 4), device="cuda"), bad,
                                     torch.zeros((1, 4), dtype=torch.int32, device="cuda"), 2)
    assert binding.spec_get_status() == 7
    assert (out[0] == -1).all()


def _keys_of(keys, tok_h, par_h, b, nodes):
    """Path keys of the given nodes of tree b (filled in as they are reached)."""
    out = []
    for u in nodes:
        u = int(u)
        if (b, u) not in keys:
            keys[(b, u)] = node_key(_keys_of(keys, tok_h, par_h, b, [par_h[b, u]])[0], int(tok_h[b, u]))
        out.append(keys[(b, u)])
    return out


def _grow_gpu(w, B):
    M = w.M
    tok = torch.zeros((B, M), dtype=torch.int32, device="cuda")
    val = torch.zeros((B, M), dtype=torch.float32, device="cuda")
    par = torch.zeros((B, M), dtype=torch.int32, device="cuda")
    val[:, 0], par[:, 0] = 1.0, -1
    keys = {(b, 0): root_key(w, b) for b in range(B)}
    frontier = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    for d in range(w.depth):
        F = frontier.shape[1]
        fr, tok_h, par_h = frontier.cpu().numpy(), tok.cpu().numpy(), par.cpu().numpy()
        ks = [k for b in range(B) for k in _keys_of(keys, tok_h, par_h, b, fr[b])]
        rows = draft_rows(w, ks, "cuda").view(B, F, w.V)
        kn = w.k if d < w.depth - 1 else 0
        frontier = binding.spec_eagle2_expand(rows, frontier, tok, val, par, w.k, w.offset(d), kn, w.T)
        assert binding.spec_get_status() == 0
    return tok, val, par


def _grow_oracle(w, B):
    M = w.M
    tok = np.zeros((B, M), np.int32)
    val = np.zeros((B, M), np.float64)
    par = np.zeros((B, M), np.int32)
    val[:, 0], par[:, 0] = 1.0, -1
    keys = {(b, 0): root_key(w, b) for b in range(B)}
    near = np.zeros(B, bool)
    frontier = np.zeros((B, 1), np.int32)
    for d in range(w.depth):
        F = frontier.shape[1]
        ks = [k for b in range(B) for k in _keys_of(keys, tok, par, b, frontier[b])]
        rows = draft_rows(w, ks, "cpu")
        tt, tp = oracle.topk_prob(rows, w.k, w.T)
        kn = w.k if d < w.depth - 1 else 0
        frontier, nr = oracle.eagle2_expand(frontier, tt.reshape(B, F, w.k), tp.reshape(B, F, w.k), tok, val, par,
                                            w.offset(d), kn)
        near |= nr
    return tok, val, par, near


def _budget_parity(w, B):
    tok, val, par = _grow_gpu(w, B)
    otok, oval, opar, near = _grow_oracle(w, B)
    op, ot, oi = binding.spec_eagle2_rerank(val, par, tok, w.m)
    assert binding.spec_get_status() == 0
    rp, rt, ri, rnear = oracle.eagle2_rerank(oval, opar, otok, w.m)
    near |= rnear
    same_tree = (tok.cpu().numpy() == otok).all(1) & (par.cpu().numpy() == opar).all(1)
    same_keep = ((op.cpu().numpy() == rp).all(1) & (ot.cpu().numpy() == rt).all(1) &
                 (oi.cpu().numpy() == ri).all(1))
    ok = same_tree & same_keep
    record_parity("eagle2", ok, near, B * w.m, "(EAGLE-2 trees, selection boundary)")
    v = val.cpu().numpy()[same_tree]
    np.testing.assert_allclose(v, oval[same_tree], rtol=1e-5, atol=0)
    return int(near.sum())


BUDGETS = [(4, 32000, "f32", 1.0, 4, 3, 12), (6, 4096, "bf16", 0.8, 8, 4, 30), (3, 128256, "bf16", 1.0, 10, 3, 40),
           (5, 1000, "f32", 1.2, 16, 2, 100), (8, 50, "bf16", 1.0, 3, 6, 20), (2, 20000, "f32", 1.0, 32, 2, 200)]


@pytest.mark.parametrize("B,V,dtype,T,k,depth,m", BUDGETS,
                         ids=[f"B{c[0]}V{c[1]}{c[2]}k{c[4]}D{c[5]}m{c[6]}" for c in BUDGETS])
def test_budget_loop_parity(B, V, dtype, T, k, depth, m):
    w = Eagle2Workload("t", B=B, V=V, dtype=dtype, T=T, k=k, depth=depth, m=m, data_seed=B * 13 + V)
    _budget_parity(w, B)


def test_budget_workload_full_size():
    w = EAGLE2_WORKLOADS["eg1"]
    _budget_parity(w, w.B)


@pytest.mark.parametrize("M,m", [(3000, 1500), (8192, 4000)])
def test_rerank_keeps_more_nodes_than_a_thread_holds(M, m):
    """Large synthetic budgets: values are products of confidences along the
    path (a child never above its parent), so the m best nodes form a tree;
    m beyond 1024 kept nodes takes the rerank's tokens from memory for the
    ranks its threads do not hold."""
    B = 2
    rng = np.random.default_rng(M + m)
    par = np.zeros((B, M), np.int32)
    val = np.zeros((B, M), np.float32)
    tok = rng.integers(0, 50000, (B, M)).astype(np.int32)
    par[:, 0], val[:, 0] = -1, 1.0
    for b in range(B):
        for c in range(1, M):
            u = int(rng.integers(max(0, c - 40), c))
            par[b, c] = u
            val[b, c] = np.float32(val[b, u] * np.float32(rng.uniform(0.3, 1.0)))
    g_val, g_par, g_tok = (torch.from_numpy(a).cuda() for a in (val, par, tok))
    op, ot, oi = binding.spec_eagle2_rerank(g_val, g_par, g_tok, m)
    assert binding.spec_get_status() == 0
    rp, rt, ri, near = oracle.eagle2_rerank(val.astype(np.float64), par, tok, m)
    ok = (op.cpu().numpy() == rp).all(1) & (ot.cpu().numpy() == rt).all(1) & (oi.cpu().numpy() == ri).all(1)
    assert ok.all()


def test_kept_tree_feeds_the_tree_mask():
    """The rerank's listing is a valid tree (parent[c] < c) whose mask and
    depths the tree-mask kernel builds."""
    w = Eagle2Workload("t", B=3, V=2000, dtype="f32", T=1.0, k=4, depth=3, m=15, data_seed=5)
    tok, val, par = _grow_gpu(w, w.B)
    op, ot, oi = binding.spec_eagle2_rerank(val, par, tok, w.m)
    mask, depth = binding.spec_tree_mask(op)
    assert binding.spec_get_status() == 0
    p = op.cpu().numpy()
    for b in range(w.B):
        assert p[b, 0] == -1 and all(0 <= p[b, c] < c for c in range(1, w.m + 1))
        rm, rd = oracle.tree_mask(p[b])
        assert np.array_equal(depth[b].cpu().numpy(), rd)
