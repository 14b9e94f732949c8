"""Pins of the oracle's verification of point-mass drafts (a deterministic
drafter such as the n-gram drafter proposes tokens, not a distribution).

* With q the point mass at the draft token, the rule is the chain rule, so
  the result must equal the chain oracle's (pinned on its own) on draft
  logits that are one-hot (0 at the draft, -inf elsewhere): exactly, except
  sequences either side flags near a boundary (their weights are scaled
  differently, p vs exp(z - m)).  Per-sequence draft counts k equal the
  chain with K = k on the first k + 1 rows, keyed by the same sequence index.
* The lossless identity for a point mass (blog.oscine.io
  "投机解码：让大模型「猜」着跑的数学魔术", §"验收标准的精确数学"): whatever
  the drafter proposes, the first emitted token is distributed as p_0
  (chi-square over seeded trials).
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def _bf16(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _onehot(x, K, V):
    nb = x.shape[0]
    zd = np.full((nb, K, V), -np.inf, dtype=np.float32)
    for s in range(nb):
        for i in range(K):
            zd[s, i, x[s, i]] = 0.0
    return zd


@pytest.mark.parametrize("K,V,T,dtype", [(1, 50, 1.0, "f32"), (4, 300, 0.8, "f32"), (5, 257, 1.2, "bf16"),
                                         (3, 64, 0.0, "f32"), (6, 1000, 1.0, "bf16")])
def test_equals_the_chain_with_one_hot_drafts(K, V, T, dtype):
    rng = np.random.default_rng(K * 100 + V)
    nb = 300
    zt = (rng.standard_normal((nb, K + 1, V)) * 3).astype(np.float32)
    # drafts that are often the target's likely tokens, sometimes not
    x = np.where(rng.random((nb, K)) < 0.6, zt[:, :K].argmax(-1), rng.integers(0, V, (nb, K))).astype(np.int32)
    zd = _onehot(x, K, V)
    if dtype == "bf16":
        zt, zd = _bf16(zt), _bf16(zd)
    pts = oracle.verify_points(zt, x, None, T, 42)
    chain = oracle.verify_chain(zt, zd, x, T, 42)
    same = (pts["n"] == chain["n_accepted"]) & np.all(pts["tokens"] == chain["tokens"], axis=1)
    assert np.all(same | pts["near"] | chain["near"])
    assert same.mean() > 0.99


def test_draft_counts_equal_the_shorter_chain():
    rng = np.random.default_rng(7)
    nb, K, V, T = 200, 6, 200, 1.0
    zt = (rng.standard_normal((nb, K + 1, V)) * 3).astype(np.float32)
    x = np.where(rng.random((nb, K)) < 0.7, zt[:, :K].argmax(-1), rng.integers(0, V, (nb, K))).astype(np.int32)
    counts = rng.integers(0, K + 1, nb).astype(np.int32)
    x_pad = x.copy()
    for s in range(nb):
        x_pad[s, counts[s]:] = -1                  # not read past the count
    pts = oracle.verify_points(zt, x_pad, counts, T, 9)
    for s in range(nb):
        k = int(counts[s])
        ch = oracle.verify_chain(zt[s:s + 1, :k + 1], _onehot(x[s:s + 1, :k], k, V), x[s:s + 1, :k], T, 9,
                                 b_ids=np.array([s]))
        if pts["near"][s] or ch["near"][0]:
            continue
        assert pts["n"][s] == ch["n_accepted"][0]
        assert pts["tokens"][s, :k + 1].tolist() == ch["tokens"][0].tolist()
        assert np.all(pts["tokens"][s, k + 1:] == -1)


def test_first_token_is_distributed_as_p():
    """V = 6, one fixed draft token at position 0: P(first token = v) = p_0(v)."""
    rng = np.random.default_rng(11)
    V, nb = 6, 300000
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = np.exp(row.astype(np.float64) - row.max())
    p /= p.sum()
    zt = np.empty((nb, 2, V), np.float32)
    zt[:, 0] = row
    zt[:, 1] = rng.standard_normal(V).astype(np.float32)
    x = np.full((nb, 1), 2, np.int32)              # a token that is not the most likely
    out = oracle.verify_points(zt, x, None, 1.0, 123, nthreads=oracle.max_threads())
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    chi = ((counts - p * nb) ** 2 / (p * nb)).sum()
    assert stats.chi2.sf(chi, V - 1) > 1e-4, (counts / nb, p)


def test_bad_counts_and_tokens_mark_the_sequence():
    zt = np.zeros((3, 4, 10), np.float32)
    x = np.array([[1, 2, 3], [1, 20, 3], [1, 2, 3]], np.int32)
    out = oracle.verify_points(zt, x, np.array([3, 3, 4], np.int32), 1.0, 0)
    assert out["status"] == oracle.ERR_TOKEN
    assert out["n"].tolist()[1:] == [-1, -1] and out["n"][0] >= 0
    ok = oracle.verify_points(zt, x, np.array([3, 1, 0], np.int32), 1.0, 0)   # the bad token is past the count
    assert ok["status"] == oracle.OK and ok["n"][1] <= 1 and ok["n"][2] == 0
