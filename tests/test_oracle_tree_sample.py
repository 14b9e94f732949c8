"""Pins of the oracle's stochastic tree verification (candidates of a node are
tried sibling by sibling; a reject replaces the target distribution r by
norm(max(0, r - q)); an accepted leaf draws a bonus from its own p).

The pages give the chain rule but not the rule for several children of one
node (infra-guide "5.3 Medusa, EAGLE và MTP", §9: verifying a tree does not by
itself keep the output lossless).  The reading is pinned by what it must
satisfy, not by its own formula:
  * a chain-shaped tree is exactly the chain verification of the same rows
    (the chain oracle is pinned on its own);
  * the lossless identity of blog.oscine.io "投机解码：让大模型「猜」着跑的数学魔术",
    §"验收标准的精确数学": with candidates drawn independently from q, the
    first emitted token is distributed as p at the root, and after an accepted
    candidate the next token as p at that candidate (chi-square over seeded
    trials);
  * hand cases of the residual recurrence with injected uniforms.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def _chain_parent(K):
    return np.array([-1] + list(range(K)), dtype=np.int32)


@pytest.mark.parametrize("K,V,T,sd,dtype", [(1, 50, 1.0, 1.0, "f32"), (4, 300, 0.8, 0.5, "f32"),
                                            (5, 257, 1.2, 3.0, "bf16"), (8, 64, 1.0, 0.05, "f32"),
                                            (0, 40, 1.0, 1.0, "f32")])
def test_chain_shaped_tree_is_the_chain(K, V, T, sd, dtype):
    rng = np.random.default_rng(K * 1000 + V)
    nb = 200
    zt = (rng.standard_normal((nb, K + 1, V)) * 3).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((nb, K, V)) * sd).astype(np.float32)
    if dtype == "bf16":  # the same values as bfloat16 bit patterns
        zt = (zt.view(np.uint32) >> 16).astype(np.uint16)
        zd = (zd.view(np.uint32) >> 16).astype(np.uint16)
    x = rng.integers(0, V, (nb, K)).astype(np.int32)
    chain = oracle.verify_chain(zt, zd, x, T, 77)
    # tree: node c (c >= 1) is draft c - 1; draft row u is the draft at node u
    # (the leaf's draft row is never read: any values)
    zd_tree = np.concatenate([zd, zd[:, :1]], axis=1) if K > 0 else zt.copy()
    tok = np.concatenate([np.zeros((nb, 1), np.int32), x], axis=1)
    tree = oracle.verify_tree_sample(zt, zd_tree, _chain_parent(K), tok, T, 77)
    assert np.array_equal(tree["length"], chain["n_accepted"] + 1)
    assert np.array_equal(tree["path"], chain["tokens"])
    assert np.array_equal(tree["near"], chain["near"])
    assert np.array_equal(tree["fallback"], chain["fallback"])


def _softmax(z, T):
    a = z.astype(np.float64) / T
    a -= a.max()
    e = np.exp(a)
    return e / e.sum()


def _chi2_ok(counts, probs, n):
    exp = probs * n
    keep = exp > 5
    chi = ((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum() + \
        (counts[~keep].sum() - exp[~keep].sum()) ** 2 / max(exp[~keep].sum(), 1e-9)
    dof = int(keep.sum())
    return stats.chi2.sf(chi, dof) > 1e-4


def test_first_token_is_distributed_as_p_at_the_root():
    """Root with 3 leaf candidates drawn i.i.d. from q: P(first token) = p."""
    rng = np.random.default_rng(5)
    V, T, nb = 6, 1.0, 400000
    parent = np.array([-1, 0, 0, 0], dtype=np.int32)
    zt_root = (rng.standard_normal(V) * 1.5).astype(np.float32)
    zd_root = (zt_root + rng.standard_normal(V) * 1.0).astype(np.float32)
    zt_leaf = (rng.standard_normal((3, V))).astype(np.float32)
    p, q = _softmax(zt_root, T), _softmax(zd_root, T)
    zt = np.empty((nb, 4, V), np.float32)
    zt[:, 0] = zt_root
    zt[:, 1:] = zt_leaf
    zd = np.empty((nb, 4, V), np.float32)
    zd[:] = zd_root
    tok = np.zeros((nb, 4), np.int32)
    tok[:, 1:] = rng.choice(V, size=(nb, 3), p=q)
    out = oracle.verify_tree_sample(zt, zd, parent, tok, T, 2024, nthreads=oracle.max_threads())
    first = out["path"][:, 0]
    assert first.min() >= 0
    counts = np.bincount(first, minlength=V)
    assert _chi2_ok(counts, p, nb), (counts / nb, p)


def test_next_token_after_an_accepted_candidate_is_p_there():
    """Depth 2: root -> 2 candidates -> 2 candidates each.  Rows of a node depend
    on its token only (identical contexts give identical rows); given the
    root's candidate with token v was accepted, the next emitted token follows
    p at v."""
    rng = np.random.default_rng(9)
    V, T, nb = 5, 0.9, 400000
    parent = np.array([-1, 0, 0, 1, 1, 2, 2], dtype=np.int32)
    t_root = (rng.standard_normal(V) * 1.5).astype(np.float32)
    d_root = (t_root + rng.standard_normal(V)).astype(np.float32)
    t_tab = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)   # target row after token v
    d_tab = (t_tab + rng.standard_normal((V, V))).astype(np.float32)  # draft row after token v
    leaf_t = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)   # rows of the leaves (unused by the test)
    tok = np.zeros((nb, 7), np.int32)
    tok[:, 1:3] = rng.choice(V, size=(nb, 2), p=_softmax(d_root, T))
    zt = np.empty((nb, 7, V), np.float32)
    zd = np.empty((nb, 7, V), np.float32)
    zt[:, 0], zd[:, 0] = t_root, d_root
    for c in (1, 2):
        v = tok[:, c]
        zt[:, c], zd[:, c] = t_tab[v], d_tab[v]
        for g in (2 * c + 1, 2 * c + 2):
            # grandchildren drawn from q at their parent
            qp = np.stack([_softmax(d_tab[w], T) for w in range(V)])
            u = rng.random(nb)
            tok[:, g] = (qp[v].cumsum(axis=1) < u[:, None]).sum(axis=1).clip(0, V - 1)
            zt[:, g] = leaf_t[tok[:, g]]
            zd[:, g] = leaf_t[tok[:, g]]
    out = oracle.verify_tree_sample(zt, zd, parent, tok, T, 99, nthreads=oracle.max_threads())
    path, length = out["path"], out["length"]
    assert _chi2_ok(np.bincount(path[:, 0], minlength=V), _softmax(t_root, T), nb)
    for v in range(V):
        sel = (length >= 2) & (path[:, 0] == v)
        n = int(sel.sum())
        if n < 2000:
            continue
        assert _chi2_ok(np.bincount(path[sel, 1], minlength=V), _softmax(t_tab[v], T), n), v


def _rows(prob_rows):
    return np.log(np.asarray(prob_rows, dtype=np.float64)).astype(np.float32)


def test_hand_cases_of_the_residual_recurrence():
    """V = 3, root with two leaf candidates; p = (0.5, 0.3, 0.2), q = (0.2, 0.6, 0.2)
    at the root (T = 1).  After the first reject r1 = max(0, p - q)/0.3 =
    (1, 0, 0); a second candidate x is then accepted iff u < r1(x)/q(x)."""
    parent = np.array([-1, 0, 0], dtype=np.int32)
    zt = _rows([[0.5, 0.3, 0.2], [0.1, 0.1, 0.8], [0.7, 0.2, 0.1]])[None]
    zd = _rows([[0.2, 0.6, 0.2], [1 / 3] * 3, [1 / 3] * 3])[None]

    def run(tok, ua, us):
        u_acc = np.zeros((1, 3))
        u_samp = np.zeros((1, 3))
        u_acc[0, 1:] = ua
        u_samp[0] = us
        out = oracle.verify_tree_sample(zt, zd, parent, np.array([[0] + tok], np.int32), 1.0, 0,
                                        u_acc=u_acc, u_samp=u_samp)
        L = out["length"][0]
        return out["path"][0, :L].tolist()

    # first candidate (token 1): p/q = 0.5 -> accepted under u = 0.4; leaf 1 draws
    # its bonus from (0.1, 0.1, 0.8): t = 0.5 falls in token 2
    assert run([1, 1], [0.4, 0.0], [0.0, 0.5, 0.0]) == [1, 2]
    # rejected under u = 0.6; second candidate token 1: r1(1) = 0 -> rejected for
    # any u; the residual after two rejects is (0.24, 0, 0) -> token 0
    assert run([1, 1], [0.6, 0.0], [0.99, 0.0, 0.0]) == [0]
    # second candidate token 0: r1(0)/q(0) = 1/0.2 = 5 -> accepted; leaf 2's
    # bonus from (0.7, 0.2, 0.1) at t = 0.8 -> token 1
    assert run([1, 0], [0.6, 0.999], [0.0, 0.0, 0.8]) == [0, 1]
    # second candidate token 2: r1(2) = 0 -> rejected; draw from (0.24, 0, 0)
    assert run([1, 2], [0.6, 0.0], [0.3, 0.0, 0.0]) == [0]


def test_all_tokens_checked_and_parent_validated():
    zt = np.zeros((2, 3, 4), np.float32)
    zd = np.zeros((2, 3, 4), np.float32)
    parent = np.array([-1, 0, 0], dtype=np.int32)
    tok = np.array([[0, 1, 2], [0, 1, 4]], np.int32)
    out = oracle.verify_tree_sample(zt, zd, parent, tok, 1.0, 0)
    assert out["status"] == oracle.ERR_TOKEN
    assert out["length"][1] == -1 and np.all(out["path"][1] == -1)
    assert out["length"][0] >= 1
    with pytest.raises(ValueError):
        oracle.verify_tree_sample(zt, zd, np.array([-1, 1, 0], np.int32), tok, 1.0, 0)
