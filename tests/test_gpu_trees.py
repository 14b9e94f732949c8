"""GPU parity of tree verification with one tree per sequence
(spec_verify_trees_greedy / spec_verify_trees, parent [B, N]) against the
oracle run sequence by sequence with its own tree (and, for the stochastic
form, its own sequence index for the uniforms): random trees that differ
between sequences, and the trees the EAGLE-2 budget keeps."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import Eagle2Workload, gumbel_argmax_draws

from gpu_helpers import NTHREADS, record_parity

pytestmark = pytest.mark.gpu


def _random_parents(rng, B, N, span=5):
    return np.stack([[-1] + [int(rng.integers(max(0, c - span), c)) for c in range(1, N)] for _ in range(B)]
                    ).astype(np.int32)


def _depth(par):
    d = np.zeros(len(par), np.int64)
    for c in range(1, len(par)):
        d[c] = d[par[c]] + 1
    return int(d.max())


def _inputs(B, N, V, dtype, T, seed, parents, sd=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    zt32 = torch.randn((B, N, V), generator=g, device="cuda") * 3
    zt, zd = zt32.to(tdt), (zt32 + torch.randn((B, N, V), generator=g, device="cuda") * sd).to(tdt)
    par = torch.tensor(parents, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    for b in range(B):   # candidates drawn from the draft at their parent
        rows = zd[b, par[b, 1:].long()].float() / (T if T > 0 else 1.0)
        tok[b, 1:] = gumbel_argmax_draws(rows, g)
    return zt, zd, par, tok.contiguous()


def _oracle_per_seq(zt, zd, par, tok, T, seed, D):
    B = zt.shape[0]
    paths, lens, near = [], [], []
    for b in range(B):
        p = par[b].cpu().numpy()
        if T == 0:
            pa, ln, st = oracle.verify_tree_greedy(zt[b:b + 1].cpu(), p, tok[b:b + 1].cpu(), max_depth=D)
            nr = np.zeros(1, bool)
        else:
            r = oracle.verify_tree_sample(zt[b:b + 1].cpu(), zd[b:b + 1].cpu(), p, tok[b:b + 1].cpu(), T, seed,
                                          max_depth=D, b_ids=[b], nthreads=NTHREADS)
            pa, ln, nr = r["path"], r["length"], r["near"]
        paths.append(pa[0])
        lens.append(ln[0])
        near.append(bool(nr[0]))
    return np.stack(paths), np.array(lens), np.array(near)


def _compare(path, length, rpath, rlen, near, positions, T):
    ok = (length == rlen) & np.all(path == rpath, axis=1)
    if T > 0:
        record_parity("trees", ok, near, positions)
    else:  # greedy: bit-exact
        bad = np.where(~ok)[0]
        assert bad.size == 0, f"{bad.size} greedy trees differ (first b={bad[0]})"


CASES = [(6, 9, 1000, "f32", 0.0), (5, 31, 4096, "bf16", 0.0), (4, 63, 32000, "bf16", 0.0),
         (6, 9, 1000, "f32", 1.0), (5, 31, 4096, "bf16", 0.8), (4, 63, 32000, "bf16", 1.0)]


@pytest.mark.parametrize("B,N,V,dtype,T", CASES, ids=[f"B{c[0]}N{c[1]}V{c[2]}{c[3]}T{c[4]}" for c in CASES])
def test_trees_that_differ_per_sequence(B, N, V, dtype, T):
    rng = np.random.default_rng(N * 7 + V)
    parents = _random_parents(rng, B, N)
    D = max(_depth(p) for p in parents)
    zt, zd, par, tok = _inputs(B, N, V, dtype, T, seed=N + V, parents=parents)
    if T == 0:
        path, length = binding.spec_verify_tree_greedy(zt, par, tok, max_depth=D)
    else:
        path, length = binding.spec_verify_tree(zt, zd, par, tok, T, 77, max_depth=D)
    assert binding.spec_get_status() == 0
    rpath, rlen, near = _oracle_per_seq(zt, zd, par, tok, T, 77, D)
    _compare(path.cpu().numpy(), length.cpu().numpy(), rpath, rlen, near, B * (N - 1), T)


def test_shared_tree_as_rows_matches_the_shared_call():
    """The same tree repeated in every row gives exactly the one-tree result."""
    rng = np.random.default_rng(3)
    one = _random_parents(rng, 1, 40)[0]
    B, N, V = 8, 40, 5000
    zt, zd, par, tok = _inputs(B, N, V, "bf16", 1.0, seed=9, parents=np.tile(one, (B, 1)))
    shared = torch.tensor(one, dtype=torch.int32, device="cuda")
    for T in (0.0, 1.0):
        a = binding.spec_verify_tree(zt, zd, par, tok, T, 5)
        b = binding.spec_verify_tree(zt, zd, shared, tok, T, 5)
        assert binding.spec_get_status() == 0
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_malformed_row_marks_only_its_sequence():
    rng = np.random.default_rng(4)
    parents = _random_parents(rng, 3, 12)
    parents[1, 5] = 9                       # a parent after its child
    zt, zd, par, tok = _inputs(3, 12, 300, "f32", 1.0, seed=2, parents=parents)
    path, length = binding.spec_verify_tree_greedy(zt, par, tok, max_depth=11)
    assert binding.spec_get_status() == 7
    ln = length.cpu().numpy()
    assert ln[1] == -1 and ln[0] >= 1 and ln[2] >= 1


def test_eagle2_trees_are_verified():
    """The budget's kept trees (one per sequence) through both verifications."""
    from test_gpu_eagle2 import _grow_gpu
    w = Eagle2Workload("t", B=4, V=8000, dtype="bf16", T=1.0, k=4, depth=3, m=20, data_seed=11)
    tok, val, par = _grow_gpu(w, w.B)
    op, ot, oi = binding.spec_eagle2_rerank(val, par, tok, w.m)
    assert binding.spec_get_status() == 0
    N = w.m + 1
    D = max(_depth(p) for p in op.cpu().numpy())
    g = torch.Generator(device="cuda").manual_seed(21)
    zt = (torch.randn((w.B, N, w.V), generator=g, device="cuda") * 3).to(torch.bfloat16)
    zd = (zt.float() + torch.randn((w.B, N, w.V), generator=g, device="cuda")).to(torch.bfloat16)
    ot = (ot % w.V).contiguous()            # the stand-in draft's token ids, folded into this V
    for T in (0.0, 1.0):
        path, length = binding.spec_verify_tree(zt, zd, op, ot, T, 13, max_depth=D)
        assert binding.spec_get_status() == 0
        rpath, rlen, near = _oracle_per_seq(zt, zd, op, ot, T, 13, D)
        _compare(path.cpu().numpy(), length.cpu().numpy(), rpath, rlen, near, w.B * w.m, T)
