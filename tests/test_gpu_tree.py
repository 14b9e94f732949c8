"""GPU parity of the greedy tree verification (spec_verify_tree_greedy) and of
the tree-attention mask builder (spec_tree_mask) with the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import tree_parents

from gpu_helpers import NTHREADS

pytestmark = pytest.mark.gpu


def _random_parent(rng, N):
    return [-1] + [int(rng.integers(max(0, c - 4), c)) for c in range(1, N)]


def _tree_case(B, N, V, dtype, seed, parent=None, p_correct=0.7, int_logits=False):
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    if parent is None:
        parent = _random_parent(rng, N)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if int_logits:
        zt = torch.randint(-3, 4, (B, N, V), generator=g, device="cuda").to(tdt)
    else:
        zt = (torch.randn((B, N, V), generator=g, device="cuda") * 3).to(tdt)
    amax = torch.argmax(zt.float(), dim=-1).to(torch.int32)
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    coin = torch.rand((B, N), generator=g, device="cuda") < p_correct
    tok = torch.where(coin, amax[:, par.clamp(min=0).long()],
                      torch.randint(0, V, (B, N), generator=g, device="cuda", dtype=torch.int32))
    tok[:, 0] = 0
    return zt, par, tok.contiguous(), parent


CASES = [(4, 1, 10, "f32"), (6, 5, 7, "bf16"), (8, 17, 33, "f32"), (8, 31, 4096, "bf16"),
         (5, 63, 32000, "f32"), (4, 63, 128256, "bf16"), (3, 200, 5000, "bf16"), (2, 1024, 300, "f32")]


@pytest.mark.parametrize("B,N,V,dtype", CASES, ids=[f"B{c[0]}N{c[1]}V{c[2]}{c[3]}" for c in CASES])
@pytest.mark.parametrize("int_logits", [False, True])
def test_tree_greedy_bit_exact(B, N, V, dtype, int_logits):
    zt, par, tok, parent = _tree_case(B, N, V, dtype, seed=N * 7 + V, int_logits=int_logits)
    path, length = binding.spec_verify_tree_greedy(zt, par, tok)
    assert binding.spec_get_status() == 0
    rpath, rlen, st = oracle.verify_tree_greedy(zt.cpu(), parent, tok.cpu(), nthreads=NTHREADS)
    assert st == oracle.OK
    assert np.array_equal(length.cpu().numpy(), rlen)
    assert np.array_equal(path.cpu().numpy(), rpath)


def test_page_example_tree():
    parent = [-1, 0, 0, 1, 2]
    V = 4
    zt = torch.zeros((1, 5, V), device="cuda")
    zt[0, 0, 2] = 1.0
    zt[0, 2, 3] = 1.0
    zt[0, 4, 1] = 1.0
    tok = torch.tensor([[0, 1, 2, 0, 3]], dtype=torch.int32, device="cuda")
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    path, length = binding.spec_verify_tree_greedy(zt, par, tok)
    assert length.item() == 3 and path[0].tolist() == [2, 3, 1]


def test_malformed_tree_reports_parent_error():
    zt, par, tok, parent = _tree_case(3, 8, 50, "f32", seed=1)
    bad = par.clone()
    bad[5] = 6                                  # parent after its child
    path, length = binding.spec_verify_tree_greedy(zt, bad, tok, max_depth=7)
    assert binding.spec_get_status() == 7
    assert np.all(length.cpu().numpy() == -1)


def test_tree_deeper_than_max_depth_reports_parent_error():
    # a chain of depth 5 verified with max_depth 3: every node's ancestor walk
    # must stop at the limit and mark the tree malformed
    parent = [-1, 0, 1, 2, 3, 4]
    zt, par, tok, _ = _tree_case(2, 6, 40, "f32", seed=3, parent=parent, p_correct=1.0)
    path, length = binding.spec_verify_tree_greedy(zt, par, tok, max_depth=3)
    assert binding.spec_get_status() == 7
    assert np.all(length.cpu().numpy() == -1)
    assert np.all(path.cpu().numpy() == -1)


def test_equal_depth_accepted_siblings_take_the_lowest_index():
    # nodes 1 and 2 carry the same token (the root row's argmax), and so do
    # their children 3 and 4 under their own rows: both depth-2 nodes are
    # accepted, and the path must run through the lower index (1, then 3)
    parent = [-1, 0, 0, 1, 2, 0]
    V = 16
    zt = torch.zeros((1, 6, V), device="cuda")
    zt[0, 0, 5] = 2.0       # root row: argmax 5
    zt[0, 1, 7] = 2.0       # node 1's row: argmax 7
    zt[0, 2, 7] = 2.0       # node 2's row: argmax 7
    zt[0, 3, 9] = 2.0       # node 3's row: argmax 9 (the bonus)
    zt[0, 4, 11] = 2.0      # node 4's row: argmax 11
    tok = torch.tensor([[0, 5, 5, 7, 7, 3]], dtype=torch.int32, device="cuda")
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    path, length = binding.spec_verify_tree_greedy(zt, par, tok)
    assert binding.spec_get_status() == 0
    assert length.item() == 3 and path[0].tolist() == [5, 7, 9]
    rpath, rlen, st = oracle.verify_tree_greedy(zt.cpu(), parent, tok.cpu())
    assert st == oracle.OK and rlen.tolist() == [3] and rpath[0].tolist() == [5, 7, 9]


def test_node_token_out_of_range():
    zt, par, tok, parent = _tree_case(3, 8, 50, "f32", seed=2)
    tok[1, 3] = 50
    path, length = binding.spec_verify_tree_greedy(zt, par, tok)
    assert binding.spec_get_status() == 4
    ln = length.cpu().numpy()
    assert ln[1] == -1 and ln[0] >= 1 and ln[2] >= 1


@pytest.mark.parametrize("N", [1, 5, 32, 33, 63, 200, 1024])
def test_tree_mask_matches_oracle(N):
    rng = np.random.default_rng(N)
    B = 3
    static = tree_parents((4, 3, 2, 2, 1), N)
    parents = [static if (b == 0 and len(static) == N) else _random_parent(rng, N) for b in range(B)]
    if N == 5:
        parents[0] = [-1, 0, 0, 1, 2]          # the page's example
    par = torch.tensor(parents, dtype=torch.int32, device="cuda")
    mask, depth = binding.spec_tree_mask(par)
    assert binding.spec_get_status() == 0
    words = mask.cpu().numpy().view(np.uint32)
    bits = [((words[b][:, np.arange(N) // 32] >> (np.arange(N) % 32)) & 1).astype(np.uint8)
            for b in range(B)]
    for b in range(B):
        rmask, rdepth = oracle.tree_mask(parents[b])
        assert np.array_equal(bits[b], rmask)
        assert np.array_equal(depth[b].cpu().numpy(), rdepth)
    if N == 5:
        assert bits[0][4].tolist() == [1, 0, 1, 0, 1]


def test_tree_mask_malformed():
    par = torch.tensor([[-1, 0, 0], [-1, 2, 0]], dtype=torch.int32, device="cuda")
    mask, depth = binding.spec_tree_mask(par)
    assert binding.spec_get_status() == 7
    assert depth[1].tolist() == [-1, -1, -1] and depth[0].tolist() == [0, 1, 1]
