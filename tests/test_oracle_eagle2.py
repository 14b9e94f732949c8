"""Pins of the oracle's EAGLE-2 tree budget (infra-guide "5.3 Medusa, EAGLE
và MTP", section 5.2): per-row top-k with probabilities, one expansion step,
and the rerank.

* top-k against numpy's stable argsort and scipy's softmax (ties, bf16 rows,
  masked entries);
* the page's example (a 0.95 node under a 0.1 parent) as a golden fixture:
  values are products along the path and the rerank keeps the best nodes;
* brute force on random trees: the next frontier and the kept set are the
  best candidates under (value, depth, id) ordering found by Python sorting;
  the kept set holds every ancestor of a kept node; the listing is ordered by
  depth and its parents point at the same nodes as the input tree.
"""
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("R,V,k,T,dtype", [(5, 7, 3, 1.0, "f32"), (9, 1000, 10, 1.0, "f32"),
                                           (4, 4096, 16, 0.7, "bf16"), (3, 50, 50, 1.3, "f32"),
                                           (6, 33, 1, 2.0, "bf16")])
def test_topk_against_argsort_and_softmax(R, V, k, T, dtype):
    rng = np.random.default_rng(R * 31 + V)
    z = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    z[:, ::5] = np.round(z[:, ::5])          # plenty of exact ties
    z[0, : V // 3] = -np.inf                 # a masked stretch
    if dtype == "bf16":
        bits = _bf16_bits(z)
        zin, zval = bits, _bf16_values(bits)
    else:
        zin, zval = z, z
    tok, prob = oracle.topk_prob(zin, k, T)
    zd = zval.astype(np.float64)
    for r in range(R):
        order = np.argsort(-zd[r], kind="stable")[:k]   # ties: lower index first
        assert tok[r].tolist() == order.tolist()
        p = softmax(zd[r] / T)
        np.testing.assert_allclose(prob[r], p[order], rtol=1e-12, atol=0)


def _fixture():
    nodes, values, keep = [], {}, {}
    for line in open(os.path.join(HERE, "golden", "infra53_eagle2_budget.txt"), encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        kind, *f = line.split()
        if kind == "node":
            nodes.append((f[0], f[1], float(f[2])))
        elif kind == "value":
            values[f[0]] = float(f[1])
        elif kind == "keep":
            keep[int(f[0])] = f[1:]
    return nodes, values, keep


def test_page_example_values_and_rerank():
    """Builds the fixture's tree with two expansion steps and reranks it."""
    nodes, values, keep = _fixture()
    names = {n: i + 1 for i, (n, _, _) in enumerate(nodes)}   # token id of each node
    cap = 1 + 2 + 2
    tok = np.zeros((1, cap), np.int32)
    val = np.zeros((1, cap), np.float64)
    par = np.zeros((1, cap), np.int32)
    val[0, 0], par[0, 0] = 1.0, -1
    level1 = [(n, c) for n, p, c in nodes if p == "root"]
    nxt, _ = oracle.eagle2_expand(np.array([[0]]), np.array([[[names[n] for n, _ in level1]]]),
                                  np.array([[[c for _, c in level1]]]), tok, val, par, 1, 2)
    frontier = nxt[0].tolist()
    kids = []
    for u in frontier:   # one child each, in frontier order
        parent_name = [n for n in names if names[n] == tok[0, u]][0]
        kids += [(n, c) for n, p, c in nodes if p == parent_name]
    oracle.eagle2_expand(np.array([frontier]), np.array([[[names[n]] for n, _ in kids]]),
                         np.array([[[c] for _, c in kids]]), tok, val, par, 3, 0)
    by_name = {n: int(np.where(tok[0] == names[n])[0][0]) for n in names}
    for n, v in values.items():
        assert val[0, by_name[n]] == pytest.approx(v, rel=1e-12)
    for m, want in keep.items():
        op, ot, oi, near = oracle.eagle2_rerank(val, par, tok, m)
        assert not near[0]
        kept = [n for n in names if by_name[n] in oi[0, 1:].tolist()]
        assert sorted(kept, key=lambda n: -val[0, by_name[n]]) == want
        assert ot[0, 0] == 0 and op[0, 0] == -1


def _grow(rng, B, D, k, k_first, V=50, ties=False):
    """Random trees grown by the oracle's expansion with random top-k lists;
    returns the node arrays and the per-step frontiers and near flags."""
    cap = 1 + k_first * k + (D - 1) * k * k if D > 1 else 1 + k
    tok = np.zeros((B, cap), np.int32)
    val = np.zeros((B, cap), np.float64)
    par = np.zeros((B, cap), np.int32)
    val[:, 0], par[:, 0] = 1.0, -1
    frontier = np.zeros((B, 1), np.int32)
    offset, steps = 1, []
    for d in range(D):
        F = frontier.shape[1]
        probs = rng.dirichlet(np.ones(V), size=(B, F))
        if ties:
            probs = np.round(probs * 8) / 64 + 1e-3
        order = np.argsort(-probs, axis=2, kind="stable")[:, :, :k]
        tt = order.astype(np.int32)
        tp = np.take_along_axis(probs, order, axis=2)
        k_next = k_first if d == 0 else k
        if d == D - 1:
            k_next = 0
        before = val.copy()
        nxt, near = oracle.eagle2_expand(frontier, tt, tp, tok, val, par, offset, k_next)
        steps.append((frontier.copy(), tt, tp, offset, nxt, near, before))
        offset += F * k
        frontier = nxt
    return tok[:, :offset], val[:, :offset], par[:, :offset], steps


@pytest.mark.parametrize("B,D,k,k_first,ties", [(40, 4, 3, 3, False), (30, 5, 4, 2, False), (30, 3, 5, 5, True),
                                                (20, 1, 6, 6, False)])
def test_expansion_by_brute_force(B, D, k, k_first, ties):
    rng = np.random.default_rng(B * 7 + D)
    tok, val, par, steps = _grow(rng, B, D, k, k_first, ties=ties)
    for frontier, tt, tp, offset, nxt, near, before in steps:
        F = frontier.shape[1]
        for b in range(B):
            cands = []
            for f in range(F):
                u = frontier[b, f]
                for j in range(k):
                    c = offset + f * k + j
                    assert tok[b, c] == tt[b, f, j] and par[b, c] == u
                    # the value is the parent's times the probability: at every
                    # depth, the product of the probabilities on the path
                    assert val[b, c] == before[b, u] * tp[b, f, j]
                    cands.append((-val[b, c], c))
            best = [c for _, c in sorted(cands)[:nxt.shape[1]]]
            assert nxt[b].tolist() == best
            kn = nxt.shape[1]
            if 0 < kn < len(cands):
                ranked = sorted(cands)
                last = -ranked[kn - 1][0]
                expect = any(abs(-v - last) <= 1e-5 * last for v, _ in ranked[kn:])
                assert near[b] == expect


def _depths(par):
    d = np.zeros(par.shape, np.int64)
    for c in range(1, par.shape[0]):
        d[c] = d[par[c]] + 1
    return d


def _path(par, tok, c):
    out = []
    while c != -1 and c != 0:
        out.append(int(tok[c]))
        c = int(par[c])
    return out[::-1]


@pytest.mark.parametrize("B,D,k,k_first,m,ties", [(40, 4, 3, 3, 10, False), (30, 5, 4, 2, 25, False),
                                                  (30, 3, 5, 5, 40, True), (10, 2, 3, 3, 12, False),
                                                  (10, 3, 2, 2, 0, False)])
def test_rerank_by_brute_force(B, D, k, k_first, m, ties):
    rng = np.random.default_rng(B * 11 + m)
    tok, val, par, _ = _grow(rng, B, D, k, k_first, ties=ties)
    op, ot, oi, near = oracle.eagle2_rerank(val, par, tok, m)
    for b in range(B):
        dep = _depths(par[b])
        keyed = sorted(range(1, val.shape[1]), key=lambda c: (-val[b, c], dep[c], c))
        kept = set(keyed[:m])
        assert oi[b, 0] == 0 and set(oi[b, 1:].tolist()) == kept
        for c in kept:                               # ancestor-closed
            u = par[b, c]
            assert u == 0 or u in kept
        ld = dep[oi[b]]
        assert np.all(np.diff(ld) >= 0)              # listed by depth
        for i in range(1, m + 1):                    # same token paths after remapping
            assert 0 <= op[b, i] < i
            assert _path(op[b], ot[b], i) == _path(par[b], tok[b], oi[b, i])
        if 0 < m < val.shape[1] - 1:
            v_last, v_next = val[b, keyed[m - 1]], val[b, keyed[m]]
            if abs(v_last - v_next) <= 1e-5 * v_last:
                assert near[b]


def test_rerank_rejects_malformed_trees():
    val = np.array([[1.0, 0.5, 0.6]])
    tok = np.zeros((1, 3), np.int32)
    with pytest.raises(ValueError):
        oracle.eagle2_rerank(val, np.array([[-1, 0, 2]]), tok, 2)       # parent not before the child
    with pytest.raises(ValueError):
        oracle.eagle2_rerank(val, np.array([[-1, 0, 1]]), tok, 1)       # child above its parent: parent dropped
