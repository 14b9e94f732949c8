"""Pins of the oracle's draft-tree functions.

* The worked example of infra-guide, "5.3 Medusa, EAGLE và MTP", section 8:
  parents = [-1, 0, 0, 1, 2], whose tree-mask row of node 4 is
  [1, 0, 1, 0, 1] and whose siblings 1 and 2 share depth 1
  (tests/golden/infra53_tree_example.txt).
* Brute force on random tiny trees: every node's root path is checked token
  by token against numpy's argmax of its parent row, and the deepest fully
  accepted node is chosen (anhtu.dev, "Speculative Decoding: Cách LLM Sinh
  Văn Bản Nhanh Gấp 2–3 Lần", §"Token tree": the deepest accepted branch is
  the output).  Ties between equally deep nodes go to the lowest index.
* A chain is the tree 0 -> 1 -> ... -> K: greedy chain and greedy tree agree.
"""
import os

import numpy as np
import pytest

import oracle
from sampling_row_online_gb300.workloads import tree_parents

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "infra53_tree_example.txt")


def _golden():
    g = {"depth": {}}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "parents":
                g["parents"] = [int(v) for v in vals]
            elif key == "mask_row":
                g["mask_row"] = (int(vals[0]), [int(v) for v in vals[1:]])
            elif key == "depth":
                g["depth"][int(vals[0])] = int(vals[1])
    return g


def test_page_example_mask_and_depth():
    g = _golden()
    mask, depth = oracle.tree_mask(g["parents"])
    node, row = g["mask_row"]
    assert mask[node].tolist() == row
    for n, d in g["depth"].items():
        assert depth[n] == d
    # the mask is never the causal lower triangle for this tree: node 4 does
    # not see node 3, which a causal mask would show it
    assert mask[4, 3] == 0 and mask[4, 1] == 0
    assert oracle.tree_max_depth(g["parents"]) == 2


def _brute_force(argmax_rows, parent, tok):
    N = len(parent)
    best, best_depth = 0, 0
    for n in range(1, N):
        path = []
        c = n
        while c != 0:
            path.append(c)
            c = parent[c]
        if all(tok[c] == argmax_rows[parent[c]] for c in path) and len(path) > best_depth:
            best, best_depth = n, len(path)
    path = []
    c = best
    while c != 0:
        path.append(c)
        c = parent[c]
    path.reverse()
    return [tok[c] for c in path] + [argmax_rows[best]]


def _random_tree(rng, N):
    return [-1] + [int(rng.integers(0, c)) for c in range(1, N)]


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny_trees(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 9))
    V = int(rng.integers(1, 5))
    B = 3
    parent = _random_tree(rng, N)
    # small integers: ties are frequent and exercise the lowest-index rule
    zt = rng.integers(-2, 3, size=(B, N, V)).astype(np.float32)
    amax = zt.argmax(-1)                 # numpy: first index of the maximum
    tok = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        for c in range(1, N):
            tok[b, c] = amax[b, parent[c]] if rng.random() < 0.7 else rng.integers(0, V)
    D = max(0, oracle.tree_max_depth(parent))
    path, length, st = oracle.verify_tree_greedy(zt, parent, tok)
    assert st == oracle.OK
    for b in range(B):
        expect = _brute_force(amax[b], parent, tok[b])
        assert length[b] == len(expect)
        assert path[b, :len(expect)].tolist() == expect
        assert all(v == -1 for v in path[b, len(expect):D + 1])


def test_page_example_hand_logits():
    parent = [-1, 0, 0, 1, 2]
    V = 4
    zt = np.zeros((1, 5, V), dtype=np.float32)
    zt[0, 0, 2] = 1.0    # after the root the target wants token 2
    zt[0, 2, 3] = 1.0    # after node 2 it wants 3
    zt[0, 4, 1] = 1.0    # after node 4 it wants 1 (the bonus)
    tok = np.array([[0, 1, 2, 0, 3]], dtype=np.int32)    # node 1 wrong, 2 right, 4 right
    path, length, _ = oracle.verify_tree_greedy(zt, parent, tok)
    assert length[0] == 3 and path[0].tolist() == [2, 3, 1]


def test_chain_tree_equals_greedy_chain():
    rng = np.random.default_rng(3)
    K, V, B = 5, 6, 20
    zt = rng.integers(-2, 3, size=(B, K + 1, V)).astype(np.float32)
    amax = zt.argmax(-1)
    x = np.where(rng.random((B, K)) < 0.75, amax[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    res = oracle.verify_chain(zt, None, x, 0.0, seed=0)
    parent = [-1] + list(range(K))
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    path, length, _ = oracle.verify_tree_greedy(zt, parent, tok)
    for b in range(B):
        n = res["n_accepted"][b]
        assert length[b] == n + 1
        assert path[b, :n + 1].tolist() == res["tokens"][b, :n + 1].tolist()


def test_invalid_parents_rejected():
    for bad in ([0, 0], [-1, 1], [-1, 0, 3], [-1, -1]):
        assert oracle.tree_max_depth(bad) == -1
        with pytest.raises(ValueError):
            oracle.tree_mask(bad)


def test_workload_tree_shape():
    parent = tree_parents((4, 3, 2, 2, 1), 63)
    assert len(parent) == 63 and parent[0] == -1
    assert all(0 <= parent[c] < c for c in range(1, 63))
    mask, depth = oracle.tree_mask(parent)
    sizes = np.bincount(depth)
    assert sizes.tolist() == [1, 4, 12, 24, 22]
    assert oracle.tree_max_depth(parent) == 4
