"""Pins of the oracle's acceptance test, residual draw, bonus draw and the
left-to-right chain.

* Hand cases of the two regimes of the acceptance rule (blog.oscine.io,
  "投机解码：让大模型「猜」着跑的数学魔术", §"验收标准的精确数学": p >= q always
  accepts; q > p accepts with probability p/q) and of the residual
  (§"拒绝之后怎么办？——残差分布").
* The two worked narratives on the pages: four drafts with the fourth
  rejected give four tokens (anhtu.dev, "Speculative Decoding: Cách LLM Sinh
  Văn Bản Nhanh Gấp 2–3 Lần", sequence diagram under "Toán học của sự miễn
  phí"), and five drafts with the third rejected give three tokens
  (glukhov.org, "Спекулятивное декодирование", §"Конкретный пример").
* Exact enumeration on the 2^-24 uniform grid: for tiny V the probability of
  every outcome is counted exactly (the decision is monotone in u, so the
  grid is split by bisection).  The emitted token at a reached position must
  be distributed as p (the identity min(q, p) + max(0, p - q) = p of §"拒绝之后
  怎么办？" on the Oscine page), and each position must be passed with
  probability sum_x min(p(x), q(x)).  p and q in these checks come from
  scipy.special.softmax, not from the oracle.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GRID = 2 ** 24


def _f32(a):
    return np.asarray(a, dtype=np.float32)


# ---------------------------------------------------------------- hand cases
P = _f32([math.log(3.0), 0.0])      # p = (0.75, 0.25) at T = 1
Q = _f32([0.0, 0.0])                # q = (0.5, 0.5)


@pytest.mark.parametrize("scale,T", [(1.0, 1.0), (2.0, 2.0), (0.5, 0.5)])
def test_p_above_q_always_accepts(scale, T):
    for u in (0.0, 0.5, 1.0 - 2.0 ** -24):
        ok, r, _ = oracle.accept(P * scale, Q * scale, 0, T, u)
        assert ok and r == pytest.approx(1.5, rel=1e-6)


@pytest.mark.parametrize("scale,T", [(1.0, 1.0), (2.0, 2.0)])
def test_q_above_p_accepts_with_ratio(scale, T):
    ok, r, _ = oracle.accept(P * scale, Q * scale, 1, T, 0.5 - 2.0 ** -24)
    assert r == pytest.approx(0.5, rel=1e-6)
    # r is 0.5 up to the fp32 rounding of ln 3: decide on either side of it
    assert oracle.accept(P * scale, Q * scale, 1, T, r * (1 - 1e-6))[0]
    assert not oracle.accept(P * scale, Q * scale, 1, T, r * (1 + 1e-6))[0]


def test_residual_is_the_excess_of_p_over_q():
    # max(0, p - q) = (0.25, 0): every uniform draws token 0
    for u in (0.0, 0.3, 1.0 - 2.0 ** -24):
        tok, near, fb = oracle.residual_sample(P, Q, 1.0, u)
        assert tok == 0 and not fb


def test_q_zero_reads_as_infinite_ratio():
    zt = _f32([0.0, 0.0])
    zd = _f32([0.0, -np.inf])
    ok, r, _ = oracle.accept(zt, zd, 1, 1.0, 1.0 - 2.0 ** -24)
    assert ok and r == math.inf
    zt2 = _f32([0.0, -np.inf])
    ok, r, _ = oracle.accept(zt2, zd, 1, 1.0, 0.0)
    assert not ok and r == 0.0


def test_residual_zero_mass_falls_back_to_p():
    z = _f32([0.1, 0.7, -0.3])
    tok, near, fb = oracle.residual_sample(z, z, 1.0, 0.0)
    assert fb and tok == 0
    tok, near, fb = oracle.residual_sample(z, z, 1.0, 1.0 - 2.0 ** -24)
    assert fb and tok == 2


def _forced_chain(K, reject_at, V=16, resid_token=7):
    """Logits that force acceptance of drafts 0..reject_at-1 (p >= q) and a
    rejection at reject_at (target gives the draft ~0 mass and puts its mass
    on resid_token)."""
    zt = np.zeros((1, K + 1, V), dtype=np.float32)
    zd = np.zeros((1, K, V), dtype=np.float32)
    x = np.arange(1, K + 1, dtype=np.int32).reshape(1, K)
    for i in range(K):
        if i < reject_at:
            zt[0, i, x[0, i]] = 5.0          # target prefers the draft: p > q
            zd[0, i, x[0, i]] = 2.0
        elif i == reject_at:
            zt[0, i, :] = -30.0
            zt[0, i, resid_token] = 10.0     # residual concentrated on resid_token
            zd[0, i, x[0, i]] = 6.0
    return zt, zd, x


@pytest.mark.parametrize("K,reject_at", [(4, 3), (5, 2), (3, 0), (1, 0)])
def test_worked_narratives(K, reject_at):
    zt, zd, x = _forced_chain(K, reject_at)
    res = oracle.verify_chain(zt, zd, x, 1.0, seed=0, u_acc=np.full((1, K), 0.5),
                              u_samp=np.full((1, K + 1), 0.5))
    n = res["n_accepted"][0]
    assert n == reject_at
    toks = res["tokens"][0]
    assert list(toks[:n]) == list(x[0, :n])
    assert toks[n] == 7
    assert all(t == -1 for t in toks[n + 1:])
    assert (toks >= 0).sum() == reject_at + 1     # tokens emitted this iteration


def test_all_accepted_emits_bonus_from_last_target_row():
    K, V = 3, 8
    zt = np.zeros((1, K + 1, V), dtype=np.float32)
    zd = np.zeros((1, K, V), dtype=np.float32)
    x = np.array([[1, 2, 3]], dtype=np.int32)
    for i in range(K):
        zt[0, i, x[0, i]] = 4.0
    zt[0, K, :] = -50.0
    zt[0, K, 5] = 0.0
    res = oracle.verify_chain(zt, zd, x, 1.0, seed=3)
    assert res["n_accepted"][0] == K
    assert list(res["tokens"][0]) == [1, 2, 3, 5]


def test_zero_drafts_is_plain_sampling():
    zt = np.zeros((2, 1, 4), dtype=np.float32)
    zt[:, 0, 2] = 40.0
    res = oracle.verify_chain(zt, None, np.zeros((2, 0), np.int32), 1.0, seed=9)
    assert list(res["n_accepted"]) == [0, 0]
    assert res["tokens"].tolist() == [[2], [2]]


def test_token_out_of_range_is_reported():
    zt = np.zeros((2, 3, 4), dtype=np.float32)
    zd = np.zeros((2, 2, 4), dtype=np.float32)
    x = np.array([[0, 1], [4, 0]], dtype=np.int32)
    res = oracle.verify_chain(zt, zd, x, 1.0, seed=0)
    assert res["status"] == oracle.ERR_TOKEN
    assert res["n_accepted"][1] == -1 and all(res["tokens"][1] == -1)
    assert res["n_accepted"][0] >= 0


def test_greedy_chain():
    V = 6
    zt = np.zeros((1, 4, V), dtype=np.float32)
    for i, a in enumerate([2, 4, 1, 5]):
        zt[0, i, a] = 1.0
    zt[0, 1, 3] = 1.0                       # tie with 4: lowest index (3) wins
    x = np.array([[2, 4, 1]], dtype=np.int32)
    res = oracle.verify_chain(zt, None, x, 0.0, seed=0)
    assert res["n_accepted"][0] == 1
    assert list(res["tokens"][0]) == [2, 3, -1, -1]
    x2 = np.array([[2, 3, 1]], dtype=np.int32)
    res = oracle.verify_chain(zt, None, x2, 0.0, seed=0)
    assert res["n_accepted"][0] == 3 and list(res["tokens"][0]) == [2, 3, 1, 5]


def test_uniforms_are_keyed_by_sequence_position_and_slot():
    # the same draft decided at u = U(seed, b, i, 0) reproduces oracle.accept
    rng = np.random.default_rng(5)
    K, V, T, seed = 3, 12, 0.8, 77
    zt = rng.standard_normal((4, K + 1, V)).astype(np.float32)
    zd = rng.standard_normal((4, K, V)).astype(np.float32)
    x = rng.integers(0, V, (4, K)).astype(np.int32)
    res = oracle.verify_chain(zt, zd, x, T, seed, b_ids=[10, 11, 12, 13])
    for s in range(4):
        n = res["n_accepted"][s]
        for i in range(n + (1 if n < K else 0)):
            ok, _, _ = oracle.accept(zt[s, i], zd[s, i], x[s, i], T,
                                     oracle.uniform(seed, 10 + s, i, 0))
            assert ok == (i < n)
        if n < K:
            tok, _, _ = oracle.residual_sample(zt[s, n], zd[s, n], T,
                                               oracle.uniform(seed, 10 + s, n, 1))
        else:
            tok, _ = oracle.target_sample(zt[s, K], T, oracle.uniform(seed, 10 + s, K, 1))
        assert res["tokens"][s, n] == tok


# --------------------------------------------------------- exact enumeration
def _accept_count(zt, zd, x, T):
    """#{k in [0, 2^24): accept at u = k 2^-24} (accept is true for k < k*)."""
    lo, hi = 0, GRID          # invariant: accept(lo) or lo == 0; not accept(hi) or hi == GRID
    if not oracle.accept(zt, zd, x, T, 0.0)[0]:
        return 0
    if oracle.accept(zt, zd, x, T, (GRID - 1) / GRID)[0]:
        return GRID
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if oracle.accept(zt, zd, x, T, mid / GRID)[0]:
            lo = mid
        else:
            hi = mid
    return hi


def _draw_counts(draw, V):
    """Grid counts of a draw that is non-decreasing in u: counts[a] = #{k : draw(k/2^24) = a}."""
    counts = np.zeros(V, dtype=np.int64)

    def first_k_at_least(a):
        lo, hi = -1, GRID       # draw(lo) < a (virtual), draw(hi) >= a (virtual)
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if draw(mid / GRID) >= a:
                hi = mid
            else:
                lo = mid
        return hi

    starts = [first_k_at_least(a) for a in range(V)] + [GRID]
    for a in range(V):
        counts[a] = starts[a + 1] - starts[a]
    return counts


def _check_position(zt_row, zd_row, T):
    V = zt_row.size
    p = softmax(zt_row.astype(np.float64) / T)
    q = softmax(zd_row.astype(np.float64) / T)
    acc = np.array([_accept_count(zt_row, zd_row, x, T) for x in range(V)]) / GRID
    # accept probability min(1, p/q) on the 2^-24 grid
    assert np.all(np.abs(acc - np.minimum(1.0, p / q)) <= 2.0 ** -24 + 1e-12)
    res = _draw_counts(lambda u: oracle.residual_sample(zt_row, zd_row, T, u)[0], V) / GRID
    resid = np.maximum(0.0, p - q)
    if resid.sum() > 1e-12:
        assert np.all(np.abs(res - resid / resid.sum()) <= 2.0 ** -23)
    emit = q * acc + (q * (1.0 - acc)).sum() * res
    assert np.all(np.abs(emit - p) <= 2.0 ** -22), (emit, p)
    assert abs((q * acc).sum() - np.minimum(p, q).sum()) <= 2.0 ** -23


@pytest.mark.parametrize("V", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
@pytest.mark.parametrize("seed", range(3))
def test_enumerated_position_law_equals_p(V, T, seed):
    rng = np.random.default_rng(100 * V + seed)
    zt = (rng.standard_normal(V) * 1.5).astype(np.float32)
    zd = (zt + rng.standard_normal(V)).astype(np.float32)
    _check_position(zt, zd, T)


@pytest.mark.parametrize("V", [2, 4, 8])
def test_enumerated_bonus_law_equals_p(V):
    rng = np.random.default_rng(V)
    z = (rng.standard_normal(V) * 2).astype(np.float32)
    for T in (0.6, 1.0):
        cnt = _draw_counts(lambda u: oracle.target_sample(z, T, u)[0], V) / GRID
        assert np.all(np.abs(cnt - softmax(z.astype(np.float64) / T)) <= 2.0 ** -23)


@pytest.mark.parametrize("K", [1, 2, 3])
def test_enumerated_chain_reach_probabilities(K):
    """P(n >= i) = prod_{k < i} sum_x min(p_k, q_k) when x_k ~ q_k, computed by
    enumerating every draft combination and the exact grid acceptance counts."""
    V, T = 4, 1.0
    rng = np.random.default_rng(K)
    zt = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    zd = (zt[:K] + rng.standard_normal((K, V))).astype(np.float32)
    beta = []
    for i in range(K):
        q = softmax(zd[i].astype(np.float64) / T)
        acc = np.array([_accept_count(zt[i], zd[i], x, T) for x in range(V)]) / GRID
        beta.append((q * acc).sum())
        p = softmax(zt[i].astype(np.float64) / T)
        assert abs(beta[-1] - np.minimum(p, q).sum()) <= 2.0 ** -23
    # P(n = i) from the enumerated betas matches the truncated geometric law
    reach = np.cumprod([1.0] + beta)
    pn = [reach[i] * (1 - beta[i]) for i in range(K)] + [reach[K]]
    assert abs(sum(pn) - 1.0) < 1e-12
    EN = sum((i + 1) * pn[i] for i in range(K + 1))
    assert EN == pytest.approx(sum(reach), rel=1e-12)
