"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (same entry points, same geometry): every sequence of the
small workloads, sampled sequences of the large ones (the oracle recomputes
those sequences from the same bytes, keyed by their true index b)."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import WORKLOADS, make_chain, make_tree

from gpu_helpers import NTHREADS, compare_chain, compare_row_stats, gpu_chain, oracle_chain

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,nsample", [("c0", None), ("c1", None), ("c2", 48), ("c4", 24)])
def test_chain_workload(name, nsample):
    w = WORKLOADS[name]
    zt, zd, x = make_chain(w, device="cuda")
    g_tok, g_n, g_max, g_sum = gpu_chain(zt, zd, x, w.T, w.verify_seed)
    if nsample is None:
        rows = np.arange(w.B)
    else:
        rng = np.random.default_rng(0)
        rows = np.sort(np.concatenate([[0, w.B - 1], rng.choice(np.arange(1, w.B - 1), nsample - 2,
                                                                  replace=False)]))
    idx = torch.from_numpy(rows).cuda()
    ref = oracle_chain(zt[idx], zd[idx], x[idx], w.T, w.verify_seed, b_ids=rows)
    compare_chain(g_tok, g_n, ref, positions=len(rows) * w.K, rows=rows, kind=f"chain-{w.name}")
    compare_row_stats(g_max, g_sum, ref, w.T, rows=rows)
    # outputs are well formed everywhere, also outside the sample
    assert np.all((g_n >= 0) & (g_n <= w.K))
    for b in range(w.B):
        n = g_n[b]
        assert np.all(g_tok[b, n + 1:] == -1) and 0 <= g_tok[b, n] < w.V


def test_tree_workload():
    w = WORKLOADS["c3"]
    zt, parent, tok = make_tree(w, device="cuda")
    path, length = binding.spec_verify_tree_greedy(zt, parent, tok)
    assert binding.spec_get_status() == 0
    rpath, rlen, st = oracle.verify_tree_greedy(zt.cpu(), parent.cpu(), tok.cpu(), nthreads=NTHREADS)
    assert np.array_equal(length.cpu().numpy(), rlen)
    assert np.array_equal(path.cpu().numpy(), rpath)
    # the workload exercises accepted paths of several depths
    assert len(set(rlen.tolist())) >= 2


def test_greedy_chain_at_workload_size():
    w = WORKLOADS["c1"]
    zt, _, _ = make_chain(w, device="cuda", with_draft_logits=False)
    amax = torch.argmax(zt.float(), dim=-1).to(torch.int32)
    g = torch.Generator(device="cuda").manual_seed(1)
    x = torch.where(torch.rand((w.B, w.K), generator=g, device="cuda") < 0.7, amax[:, :w.K],
                    torch.randint(0, w.V, (w.B, w.K), generator=g, device="cuda",
                                  dtype=torch.int32)).contiguous()
    out, n = binding.spec_verify(zt, None, x, 0.0, 0)
    ref = oracle_chain(zt, None, x, 0.0, 0, want_stats=False)
    assert np.array_equal(n.cpu().numpy(), ref["n_accepted"])
    assert np.array_equal(out.cpu().numpy(), ref["tokens"])
