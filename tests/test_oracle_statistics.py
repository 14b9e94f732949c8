"""Statistical pins of the oracle's chain verification at scale.

* Chi-square over 10^6 seeded sequences at V = 16, K = 3: at every reached
  position the emitted token must follow p_i (the lossless property of
  blog.oscine.io, "投机解码：让大模型「猜」着跑的数学魔术", §"拒绝之后怎么办？——
  残差分布"), and the number of accepted drafts must follow
  P(n >= i) = prod_{k<i} sum_x min(p_k(x), q_k(x)).
* Expected tokens per iteration: with every position passed with the same
  probability alpha, E[N] = (1 - alpha^(K+1)) / (1 - alpha) (same page,
  §"加速比公式：什么时候值得投机？").  The worked values printed there are in
  tests/golden/oscine_expected_tokens.txt; the alpha = 0.6 line is a misprint
  (formula 2.38, printed 2.5) and the test checks the formula's value.

Draft tokens are drawn from q by the workload generator (Gumbel-max), not by
the oracle; p and q of the expected laws come from scipy.special.softmax.
"""
import os

import numpy as np
import pytest
import torch
from scipy import stats
from scipy.special import softmax

import oracle
from sampling_row_online_gb300.workloads import gumbel_argmax_draws

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "oscine_expected_tokens.txt")


def _draft_tokens(zd_rows, T, nseq, seed):
    """nseq independent draws from softmax(zd_rows[i] / T) for every position i."""
    K, V = zd_rows.shape
    g = torch.Generator().manual_seed(seed)
    scaled = torch.from_numpy(np.ascontiguousarray(
        np.broadcast_to(zd_rows.astype(np.float32) / T, (nseq, K, V)).reshape(nseq * K, V)))
    return gumbel_argmax_draws(scaled, g, chunk_rows=1 << 16).numpy().reshape(nseq, K)


def _run(zt_rows, zd_rows, T, nseq, seed):
    K = zd_rows.shape[0]
    x = _draft_tokens(zd_rows, T, nseq, seed)
    zt = np.ascontiguousarray(np.broadcast_to(zt_rows, (nseq,) + zt_rows.shape))
    zd = np.ascontiguousarray(np.broadcast_to(zd_rows, (nseq,) + zd_rows.shape))
    res = oracle.verify_chain(zt, zd, x, T, seed=seed, nthreads=max(1, os.cpu_count() or 1))
    assert res["status"] == oracle.OK
    return res


@pytest.mark.slow
def test_chisquare_million_trials_v16():
    V, K, T, nseq = 16, 3, 1.0, 10 ** 6
    rng = np.random.default_rng(2024)
    zt = (rng.standard_normal((K + 1, V)) * 1.2).astype(np.float32)
    zd = (zt[:K] + rng.standard_normal((K, V)) * 0.8).astype(np.float32)
    res = _run(zt, zd, T, nseq, seed=11)
    n, tok = res["n_accepted"], res["tokens"]
    p = softmax(zt.astype(np.float64) / T, axis=-1)
    q = softmax(zd.astype(np.float64) / T, axis=-1)
    beta = np.minimum(p[:K], q).sum(-1)
    # law of n
    reach = np.cumprod(np.concatenate([[1.0], beta]))
    pn = np.array([reach[i] * (1 - beta[i]) for i in range(K)] + [reach[K]])
    obs = np.bincount(n, minlength=K + 1)
    assert stats.chisquare(obs, pn * nseq).pvalue > 1e-3
    # law of the token emitted at each reached position
    for i in range(K + 1):
        sel = n >= i
        h = np.bincount(tok[sel, i], minlength=V)
        assert stats.chisquare(h, p[i] * sel.sum()).pvalue > 1e-3, i


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, k, c, en, s, ok = line.split()
                rows.append((float(a), int(k), float(c), float(en), float(s), ok == "1"))
    return rows


def _two_point_rows(alpha):
    """V = 2 rows with sum_x min(p, q) = alpha: p = (a, 1-a), q = (a - (1-alpha), ...)."""
    a = 0.5 + (1 - alpha) / 2
    p = np.array([a, 1 - a])
    q = np.array([a - (1 - alpha), 1 - a + (1 - alpha)])
    return np.log(p).astype(np.float32), np.log(q).astype(np.float32)


def test_expected_tokens_formula_matches_printed_values():
    for alpha, k, c, en, s, consistent in _golden_rows():
        EN = (1 - alpha ** (k + 1)) / (1 - alpha)
        S = EN / (1 + k / c)
        if consistent:
            assert round(EN, 1) == en and round(S, 1) == s
        else:
            assert round(EN, 1) != en       # the misprinted line
            assert EN == pytest.approx(2.38336, abs=1e-5) and S == pytest.approx(1.58891, abs=1e-5)


@pytest.mark.slow
@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"alpha{r[0]}")
def test_mean_tokens_per_iteration(row):
    alpha, k, c, en, s, consistent = row
    zp, zq = _two_point_rows(alpha)
    zt = np.stack([zp] * (k + 1))
    zd = np.stack([zq] * k)
    nseq = 400_000
    res = _run(zt, zd, 1.0, nseq, seed=int(alpha * 100))
    N = res["n_accepted"].astype(np.float64) + 1.0
    # alpha realised by the fp32 logits (exact to ~1e-7)
    p = softmax(zp.astype(np.float64))
    q = softmax(zq.astype(np.float64))
    a_eff = np.minimum(p, q).sum()
    EN = (1 - a_eff ** (k + 1)) / (1 - a_eff)
    se = N.std() / np.sqrt(nseq)
    assert abs(N.mean() - EN) < 5 * se
    if consistent:
        assert abs(N.mean() - en) < 0.05 + 5 * se
    else:
        assert abs(N.mean() - en) > 0.1     # the printed 2.5 is off; the formula holds
