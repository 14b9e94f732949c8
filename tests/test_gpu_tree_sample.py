"""GPU parity of the stochastic tree verification (spec_verify_tree) with the
fp64 oracle, on seeded trees whose candidates are drawn from the draft at
their parent: random trees, the static 4/3/2/2/1 tree, chain-shaped trees,
one wide node, both element types, ragged vocabularies.  Parity rule as for
the chain: path and length equal except sequences the oracle flags near a
decision boundary (their count below 1e-4 of the verified positions, one
tolerated in small tests)."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import WORKLOADS, gumbel_argmax_draws, make_tree_sample, tree_parents

from gpu_helpers import NTHREADS, record_parity

pytestmark = pytest.mark.gpu


def _random_parent(rng, N, span=4):
    return [-1] + [int(rng.integers(max(0, c - span), c)) for c in range(1, N)]


def _case(B, N, V, dtype, T, seed, parent=None, sd=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    if parent is None:
        parent = _random_parent(rng, N)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    zt32 = torch.randn((B, N, V), generator=g, device="cuda") * 3
    zd32 = zt32 + torch.randn((B, N, V), generator=g, device="cuda") * sd
    zt, zd = zt32.to(tdt), zd32.to(tdt)
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    if N > 1:
        rows = zd[:, par[1:].long()].reshape(B * (N - 1), V).float() / T
        tok[:, 1:] = gumbel_argmax_draws(rows, g).reshape(B, N - 1)
    return zt, zd, par, tok.contiguous(), parent


def _compare(path, length, ref, positions):
    ok = (length == ref["length"]) & np.all(path == ref["path"], axis=1)
    record_parity("tree_sample", ok, ref["near"], positions)


def _run(zt, zd, par, tok, parent, T, seed):
    path, length = binding.spec_verify_tree(zt, zd, par, tok, T, seed)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_tree_sample(zt.cpu(), zd.cpu(), parent, tok.cpu(), T, seed, nthreads=NTHREADS)
    assert ref["status"] == oracle.OK
    return path.cpu().numpy(), length.cpu().numpy(), ref


CASES = [(4, 1, 10, "f32", 1.0), (6, 5, 7, "bf16", 0.8), (8, 17, 33, "f32", 1.0), (8, 31, 4096, "bf16", 1.2),
         (5, 63, 32000, "f32", 1.0), (4, 63, 128256, "bf16", 0.7), (3, 200, 5000, "bf16", 1.0),
         (6, 40, 4097, "f32", 0.9)]


@pytest.mark.parametrize("B,N,V,dtype,T", CASES, ids=[f"B{c[0]}N{c[1]}V{c[2]}{c[3]}T{c[4]}" for c in CASES])
@pytest.mark.parametrize("sd", [0.3, 3.0])
def test_tree_sample_parity(B, N, V, dtype, T, sd):
    zt, zd, par, tok, parent = _case(B, N, V, dtype, T, seed=N * 13 + V, sd=sd)
    path, length, ref = _run(zt, zd, par, tok, parent, T, 4321 + N)
    _compare(path, length, ref, B * max(1, N - 1))


@pytest.mark.parametrize("V,dtype", [(257, "f32"), (32000, "bf16")])
def test_static_tree_and_a_wide_node(V, dtype):
    for parent in (tree_parents((4, 3, 2, 2, 1), 63), [-1] + [0] * 24 + list(range(1, 9))):
        zt, zd, par, tok, _ = _case(6, len(parent), V, dtype, 1.0, seed=len(parent) + V, parent=parent)
        path, length, ref = _run(zt, zd, par, tok, parent, 1.0, 99)
        _compare(path, length, ref, 6 * (len(parent) - 1))


def test_chain_shaped_tree_equals_the_chain_path():
    """parent[c] = c - 1: exactly spec_verify's result on the same rows."""
    B, K, V = 16, 5, 50257
    g = torch.Generator(device="cuda").manual_seed(3)
    zt = (torch.randn((B, K + 1, V), generator=g, device="cuda") * 3).to(torch.bfloat16)
    zd = (zt[:, :K].float() + torch.randn((B, K, V), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    x = gumbel_argmax_draws(zd.reshape(B * K, V).float() / 0.8, g).reshape(B, K)
    chain_tok, chain_n = binding.spec_verify(zt, zd, x, 0.8, 11)
    par = torch.arange(-1, K, dtype=torch.int32, device="cuda")
    zd_tree = torch.cat([zd, zd[:, :1]], dim=1).contiguous()
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), x], dim=1).contiguous()
    path, length = binding.spec_verify_tree(zt, zd_tree, par, tok, 0.8, 11)
    assert binding.spec_get_status() == 0
    assert torch.equal(length, chain_n + 1)
    assert torch.equal(path, chain_tok)


def test_zero_temperature_is_the_greedy_tree():
    zt, zd, par, tok, parent = _case(5, 31, 1000, "f32", 1.0, seed=8)
    a_path, a_len = binding.spec_verify_tree(zt, zd, par, tok, 0.0, 0)
    b_path, b_len = binding.spec_verify_tree_greedy(zt, par, tok)
    assert torch.equal(a_path, b_path) and torch.equal(a_len, b_len)


def test_errors_mark_the_sequence():
    zt, zd, par, tok, parent = _case(4, 9, 100, "f32", 1.0, seed=5)
    tok[2, 3] = 100
    path, length = binding.spec_verify_tree(zt, zd, par, tok, 1.0, 0)
    assert binding.spec_get_status() == 4
    ln = length.cpu().numpy()
    assert ln[2] == -1 and np.all(path[2].cpu().numpy() == -1) and np.all(ln[[0, 1, 3]] >= 1)
    bad = par.clone()
    bad[5] = 7
    binding.spec_verify_tree(zt, zd, bad, tok.clamp(0, 99), 1.0, 0, max_depth=8)
    assert binding.spec_get_status() == 7


def test_stochastic_tree_workload_full_size():
    w = WORKLOADS["c3s"]
    zt, zd, par, tok = make_tree_sample(w, device="cuda")
    path, length = binding.spec_verify_tree(zt, zd, par, tok, w.T, w.verify_seed)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_tree_sample(zt.cpu(), zd.cpu(), par.cpu(), tok.cpu(), w.T, w.verify_seed,
                                    nthreads=NTHREADS)
    _compare(path.cpu().numpy(), length.cpu().numpy(), ref, w.positions)
