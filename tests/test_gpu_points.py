"""GPU parity of the verification of point-mass drafts (spec_verify_points):
against the oracle with full and per-sequence draft counts, greedy and
stochastic, both element types; bit-exact against spec_verify on draft rows
that are one-hot (0 at the draft, -inf elsewhere), which the rule equals;
the n-gram drafter's output verified end to end; counts out of range."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import NgramWorkload, make_contexts

from gpu_helpers import NTHREADS, record_parity

pytestmark = pytest.mark.gpu


def _case(B, K, V, dtype, seed, p_good=0.6):
    g = torch.Generator(device="cuda").manual_seed(seed)
    zt32 = torch.randn((B, K + 1, V), generator=g, device="cuda") * 3
    zt = zt32.to(torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()
    top = zt[:, :K].float().argmax(-1).to(torch.int32)
    rnd = torch.randint(0, V, (B, K), generator=g, device="cuda", dtype=torch.int32)
    good = torch.rand((B, K), generator=g, device="cuda") < p_good
    return zt, torch.where(good, top, rnd).contiguous()


def _compare(out, n, ref, positions):
    ok = (n == ref["n"]) & np.all(out == ref["tokens"], axis=1)
    record_parity("points", ok, ref["near"], positions)


CASES = [(64, 5, 128256, "bf16", 0.7), (32, 4, 32000, "f32", 1.0), (16, 8, 4097, "bf16", 1.3),
         (64, 5, 128256, "bf16", 0.0), (40, 1, 1000, "f32", 1.0), (8, 0, 500, "f32", 1.0)]


@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("B,K,V,dtype,T", CASES, ids=[f"B{c[0]}K{c[1]}V{c[2]}{c[3]}T{c[4]}" for c in CASES])
def test_parity(B, K, V, dtype, T, ragged):
    zt, x = _case(B, K, V, dtype, seed=B * 7 + K + V)
    counts = None
    if ragged:
        counts = torch.randint(0, K + 1, (B,), dtype=torch.int32, device="cuda")
        x = torch.where(torch.arange(K, device="cuda")[None, :] < counts[:, None], x, -1).to(torch.int32)
    out, n = binding.spec_verify_points(zt, x.contiguous(), T, 31, draft_counts=counts)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_points(zt.cpu(), x.cpu(), None if counts is None else counts.cpu(), T, 31,
                               nthreads=NTHREADS)
    _compare(out.cpu().numpy(), n.cpu().numpy(), ref, B * max(K, 1))


def test_long_point_mass_chains():
    """K = 150 drafts, nearly all the target's argmax with a dominant logit:
    first rejects past position 64 (and some chains accepted whole)."""
    B, K, V, T = 16, 150, 1000, 1.0
    zt, x = _case(B, K, V, "f32", seed=77, p_good=0.99)
    top = zt[:, :K].argmax(-1, keepdim=True)
    zt[:, :K].scatter_add_(2, top, torch.full((B, K, 1), 20.0, device="cuda"))
    out, n = binding.spec_verify_points(zt, x, T, 31)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_points(zt.cpu(), x.cpu(), None, T, 31, nthreads=NTHREADS)
    _compare(out.cpu().numpy(), n.cpu().numpy(), ref, B * K)
    assert (ref["n"] >= 64).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_equals_spec_verify_on_one_hot_draft_rows(dtype):
    B, K, V = 48, 5, 50257
    zt, x = _case(B, K, V, dtype, seed=5)
    zd = torch.full((B, K, V), float("-inf"), device="cuda")
    zd.scatter_(2, x.long().unsqueeze(-1), 0.0)
    zd = zd.to(zt.dtype).contiguous()
    for T in (0.0, 0.8, 1.0):
        a = binding.spec_verify_points(zt, x, T, 77)
        b = binding.spec_verify(zt, zd, x, T, 77)
        assert binding.spec_get_status() == 0
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_ngram_drafts_end_to_end():
    """Drafts and counts from spec_ngram_propose go straight into the
    verification; target rows favour the drafted tokens."""
    w = NgramWorkload("t", B=32, L=4096, n_min=1, n_max=4, min_hits=1, K=5, data_seed=4)
    tokens, lengths = make_contexts(w, device="cuda")
    draft, count = binding.spec_ngram_propose(tokens, lengths, w.n_min, w.n_max, w.K)
    V = 128256
    g = torch.Generator(device="cuda").manual_seed(8)
    zt = torch.randn((w.B, w.K + 1, V), generator=g, device="cuda") * 2
    rows = torch.arange(w.K, device="cuda")
    has = draft >= 0
    b_idx = torch.arange(w.B, device="cuda")[:, None].expand(-1, w.K)[has]
    zt[b_idx, rows[None, :].expand(w.B, -1)[has], draft[has].long()] += 8.0   # the target agrees, mostly
    zt = zt.to(torch.bfloat16).contiguous()
    out, n = binding.spec_verify_points(zt, draft, 1.0, 3, draft_counts=count)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_points(zt.cpu(), draft.cpu(), count.cpu(), 1.0, 3, nthreads=NTHREADS)
    _compare(out.cpu().numpy(), n.cpu().numpy(), ref, w.B * w.K)
    assert (n.cpu().numpy() <= count.cpu().numpy()).all() and n.sum().item() > 0


def test_bad_counts_mark_the_sequence():
    zt, x = _case(4, 3, 100, "f32", seed=1)
    counts = torch.tensor([3, 4, -1, 0], dtype=torch.int32, device="cuda")
    out, n = binding.spec_verify_points(zt, x, 1.0, 0, draft_counts=counts)
    assert binding.spec_get_status() == 4
    nn = n.cpu().tolist()
    assert nn[1] == -1 and nn[2] == -1 and nn[0] >= 0 and nn[3] == 0
    assert (out[1:3] == -1).all()
