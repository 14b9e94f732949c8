"""Pins of the oracle's row normalisers and argmax.

The normalisers (m, S) of p = softmax(z / T) are pinned by closed forms
(constant rows, two-point rows), by the library routine
scipy.special.logsumexp (m + T ln S = T logsumexp(z / T)), and by exact
bfloat16 widening.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


@pytest.mark.parametrize("V", [1, 2, 7, 1000])
@pytest.mark.parametrize("T", [0.05, 0.7, 1.0, 3.0])
def test_constant_row(V, T):
    z = np.full(V, 2.5, dtype=np.float32)
    m, S = oracle.row_stats(z, T)
    assert m == 2.5
    assert S == pytest.approx(V, rel=1e-15)


def test_two_point_row():
    # z = [ln 3, 0] at T = 1 gives p = (3/4, 1/4): S = 1 + 1/3 relative to the max
    z = np.array([math.log(3.0), 0.0], dtype=np.float32)
    m, S = oracle.row_stats(z, 1.0)
    assert m == float(np.float32(math.log(3.0)))
    assert S == pytest.approx(1.0 + math.exp(-float(np.float32(math.log(3.0)))), rel=1e-15)
    assert 1.0 / S == pytest.approx(0.75, rel=1e-7)


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("T", [0.3, 0.7, 1.0, 2.0])
def test_against_logsumexp(seed, T):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal(5000) * 4).astype(np.float32)
    m, S = oracle.row_stats(z, T)
    assert m == float(z.max())
    lse = logsumexp(z.astype(np.float64) / T)
    assert m / T + math.log(S) == pytest.approx(lse, rel=1e-13, abs=1e-12)


def test_bf16_widening_is_exact():
    z = torch.tensor([1.0, -2.0, 0.0078125, 3.140625, -100.5], dtype=torch.bfloat16)
    m, S = oracle.row_stats(z, 1.0)
    assert m == 3.140625
    expect = sum(math.exp(float(v) - 3.140625) for v in z.float().tolist())
    assert S == pytest.approx(expect, rel=1e-15)


def test_masked_minus_inf_entries_contribute_nothing():
    z = np.array([-np.inf, 1.0, -np.inf, 1.0], dtype=np.float32)
    m, S = oracle.row_stats(z, 0.5)
    assert m == 1.0 and S == 2.0


def test_argmax_first_index_of_ties():
    assert oracle.argmax(np.array([1, 3, 3, 2], dtype=np.float32)) == 1
    assert oracle.argmax(np.array([5], dtype=np.float32)) == 0
    assert oracle.argmax(np.array([-np.inf, -1, -1], dtype=np.float32)) == 1
    zb = torch.tensor([0.5, 7.0, 7.0, 7.0], dtype=torch.bfloat16)
    assert oracle.argmax(zb) == 1
