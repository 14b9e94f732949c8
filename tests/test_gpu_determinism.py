"""Run-to-run determinism: every entry point called twice on the same inputs
gives the same bytes.  Each reduction has a fixed order and every random
number is a counter-based uniform, so a race between threads or CTAs would
show up here as drift (the check that stands in for a race detector)."""
import pytest
import torch

from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import (EAGLE2_WORKLOADS, WORKLOADS, eagle2_step_rows, make_tree_sample)

pytestmark = pytest.mark.gpu


def _twice(fn):
    a = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    b = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    assert binding.spec_get_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_stochastic_tree():
    w = WORKLOADS["c3s"]
    zt, zd, par, tok = make_tree_sample(w, device="cuda")
    _twice(lambda: binding.spec_verify_tree(zt, zd, par, tok, w.T, 5))
    pars = par.unsqueeze(0).expand(w.B, -1).contiguous()      # the same tree given per sequence
    _twice(lambda: binding.spec_verify_tree(zt, zd, pars, tok, w.T, 5))


def test_point_mass_verification():
    g = torch.Generator(device="cuda").manual_seed(2)
    B, K, V = 64, 5, 128256
    zt = (torch.randn((B, K + 1, V), generator=g, device="cuda") * 3).to(torch.bfloat16)
    x = torch.randint(0, V, (B, K), generator=g, device="cuda", dtype=torch.int32)
    counts = torch.randint(0, K + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
    _twice(lambda: binding.spec_verify_points(zt, x, 0.7, 11, draft_counts=counts))


def test_topk_and_budget():
    w = EAGLE2_WORKLOADS["eg1"]
    rows = eagle2_step_rows(w, 1, "cuda").reshape(-1, w.V)
    _twice(lambda: binding.spec_topk(rows, w.k, w.T))

    def build():
        tok = torch.zeros((w.B, w.M), dtype=torch.int32, device="cuda")
        val = torch.zeros((w.B, w.M), dtype=torch.float32, device="cuda")
        par = torch.zeros((w.B, w.M), dtype=torch.int32, device="cuda")
        val[:, 0], par[:, 0] = 1.0, -1
        front = torch.zeros((w.B, 1), dtype=torch.int32, device="cuda")
        for d in range(w.depth):
            kn = w.k if d < w.depth - 1 else 0
            front = binding.spec_eagle2_expand(eagle2_step_rows(w, d, "cuda"), front, tok, val, par, w.k,
                                               w.offset(d), kn, w.T)
        return (tok, val, par) + tuple(binding.spec_eagle2_rerank(val, par, tok, w.m))

    _twice(build)


def test_every_verification_workload_twice():
    from sampling_row_online_gb300.workloads import make_chain, make_tree
    for name in ("c0", "c1", "c3"):
        w = WORKLOADS[name]
        if w.kind == "tree":
            zt, parent, tok = make_tree(w, device="cuda")
            _twice(lambda: binding.spec_verify_tree_greedy(zt, parent, tok))
        else:
            zt, zd, x = make_chain(w, device="cuda")
            _twice(lambda: binding.spec_verify_ex(zt, zd, x, w.T, w.verify_seed, want_row_stats=True))
