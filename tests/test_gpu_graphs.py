"""The library's calls inside CUDA graphs: captured once (after a warm-up
call that sizes the stream's workspace), replayed with new input contents
copied into the captured tensors, and compared with eager calls on the same
inputs (bit-identical: the same kernels, the same uniforms).  The side stream
waits for the default stream before its first call: tensors made there may
still be in flight, and their blocks may still be in use by queued kernels."""
import pytest
import torch

from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import (Eagle2Workload, NgramWorkload, Workload, eagle2_step_rows,
                                                 make_chain, make_contexts)

pytestmark = pytest.mark.gpu


def _capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def test_chain_verification_in_a_graph():
    s = torch.cuda.Stream()
    w = Workload("g", "chain", B=16, K=5, V=32000, dtype="bf16", T=0.8, data_seed=31)
    zt, zd, x = make_chain(w, device="cuda")
    out = torch.empty((w.B, w.K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((w.B,), dtype=torch.int32, device="cuda")
    s.wait_stream(torch.cuda.current_stream())      # inputs and outputs were made on the default stream
    with torch.cuda.stream(s):
        binding.spec_verify(zt, zd, x, w.T, 9, out_tokens=out, out_n_accepted=n, stream=s)   # sizes the workspace
    s.synchronize()
    g = _capture(lambda: binding.spec_verify(zt, zd, x, w.T, 9, out_tokens=out, out_n_accepted=n, stream=s), s)
    for seed in (32, 33):
        w2 = Workload("g", "chain", B=16, K=5, V=32000, dtype="bf16", T=0.8, data_seed=seed)
        a, b, c = make_chain(w2, device="cuda")
        zt.copy_(a), zd.copy_(b), x.copy_(c)
        g.replay()
        torch.cuda.synchronize()
        assert binding.spec_get_status(s) == 0
        ref_out, ref_n = binding.spec_verify(a, b, c, w.T, 9)
        assert torch.equal(out, ref_out) and torch.equal(n, ref_n)


def test_ngram_draft_and_point_verification_in_one_graph():
    s = torch.cuda.Stream()
    V = 32000                               # the contexts' and the target's vocabulary
    w = NgramWorkload("g", B=16, L=8192, n_min=1, n_max=4, min_hits=1, K=5, V=V, data_seed=41)
    tokens, lengths = make_contexts(w, device="cuda")
    zt = (torch.randn((w.B, w.K + 1, V), device="cuda") * 3).to(torch.bfloat16)
    draft = torch.empty((w.B, w.K), dtype=torch.int32, device="cuda")
    count = torch.empty((w.B,), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((w.B,), dtype=torch.int32, device="cuda")

    def step():
        binding.spec_ngram_propose(tokens, lengths, w.n_min, w.n_max, w.K, out_draft=draft, out_count=count,
                                   stream=s)
        binding.spec_verify_points(zt, draft, 1.0, 4, draft_counts=count, out_tokens=out, out_n=n, stream=s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = _capture(step, s)
    for seed in (42, 43):
        w2 = NgramWorkload("g", B=16, L=8192, n_min=1, n_max=4, min_hits=1, K=5, V=V, data_seed=seed)
        t2, l2 = make_contexts(w2, device="cuda")
        tokens.copy_(t2), lengths.copy_(l2)
        zt.copy_((torch.randn((w.B, w.K + 1, V), device="cuda") * 3).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert binding.spec_get_status(s) == 0
        d2, c2 = binding.spec_ngram_propose(t2, l2, w.n_min, w.n_max, w.K)
        o2, n2 = binding.spec_verify_points(zt, d2, 1.0, 4, draft_counts=c2)
        assert torch.equal(draft, d2) and torch.equal(count, c2)
        assert torch.equal(out, o2) and torch.equal(n, n2)


def test_eagle2_budget_in_a_graph():
    s = torch.cuda.Stream()
    w = Eagle2Workload("g", B=4, V=8000, dtype="bf16", T=1.0, k=4, depth=3, m=12, data_seed=51)
    rows = [eagle2_step_rows(w, d, "cuda") for d in range(w.depth)]
    tok = torch.zeros((w.B, w.M), dtype=torch.int32, device="cuda")
    val = torch.zeros((w.B, w.M), dtype=torch.float32, device="cuda")
    par = torch.zeros((w.B, w.M), dtype=torch.int32, device="cuda")
    val[:, 0], par[:, 0] = 1.0, -1
    fronts = [torch.zeros((w.B, 1), dtype=torch.int32, device="cuda")] + \
             [torch.empty((w.B, w.k), dtype=torch.int32, device="cuda") for _ in range(w.depth)]
    kept = [torch.empty((w.B, w.m + 1), dtype=torch.int32, device="cuda") for _ in range(3)]

    def build():
        for d in range(w.depth):
            kn = w.k if d < w.depth - 1 else 0
            binding.spec_eagle2_expand(rows[d], fronts[d], tok, val, par, w.k, w.offset(d), kn, w.T,
                                       out_frontier=fronts[d + 1][:, :kn] if kn else fronts[d + 1][:, :0],
                                       stream=s)
        res = binding.spec_eagle2_rerank(val, par, tok, w.m, stream=s)
        for dst, src in zip(kept, res):
            dst.copy_(src)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        build()
    s.synchronize()
    first = [t.clone() for t in kept]
    g = _capture(build, s)
    g.replay()
    torch.cuda.synchronize()
    assert binding.spec_get_status(s) == 0
    assert all(torch.equal(a, b) for a, b in zip(first, kept))
