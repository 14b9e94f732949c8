"""GPU parity of the n-gram (prompt-lookup) drafter (spec_ngram_propose) with
the oracle: bit-exact drafts and counts on seeded contexts: repetitive
code-editing-like contexts, tiny alphabets (many overlapping matches), runs
of one token, the page's worked example, ragged and degenerate lengths,
unaligned rows (the scalar-load variant), batch sizes from one sequence
(hundreds of CTAs each) to a thousand (one CTA each), forced CTA counts,
min_hits > 1, and the two full-size drafting workloads."""
import os

import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import NGRAM_WORKLOADS, NgramWorkload, make_contexts

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _check(tokens, lengths, n_min, n_max, K, min_hits=1):
    """tokens may be a non-contiguous-storage view (offset rows): the kernel
    reads it through its data pointer with row stride L."""
    draft, count = binding.spec_ngram_propose(tokens, lengths, n_min, n_max, K, min_hits=min_hits)
    assert binding.spec_get_status() == 0
    ref_d, ref_c = oracle.ngram_propose(tokens.cpu().numpy(), lengths.cpu().numpy(), n_min, n_max, K,
                                        min_hits=min_hits)
    c = count.cpu().numpy()
    d = draft.cpu().numpy()
    bad = np.where((c != ref_c) | np.any(d != ref_d, axis=1))[0]
    assert bad.size == 0, (f"{bad.size} rows differ; first b={bad[0]}: gpu {c[bad[0]]} {d[bad[0]].tolist()} "
                           f"oracle {ref_c[bad[0]]} {ref_d[bad[0]].tolist()}")
    return c


# min_hits == 1 keeps a running maximum key; min_hits > 1 a histogram, in
# registers when n_max - n_min < 8 and in shared memory otherwise; L % 4 != 0
# takes the scalar loads
SHAPES = [(1, 7, 1, 4, 5, 1), (3, 64, 1, 4, 5, 1), (8, 1000, 2, 6, 8, 1), (16, 4097, 1, 3, 5, 2),
          (5, 30001, 1, 12, 6, 1), (2, 200000, 1, 4, 5, 1), (1, 1 << 20, 3, 8, 48, 1), (300, 2048, 1, 4, 5, 3),
          (4, 4096, 8, 8, 5, 2), (2, 5000, 1, 64, 255, 1), (64, 10000, 1, 4, 0, 1), (8, 8192, 1, 16, 5, 2),
          (6, 12003, 2, 40, 7, 2), (1, 300000, 1, 8, 5, 4),
          # min_hits == 1 in a cluster, drafts longer than a warp's lanes
          (8, 3001, 1, 4, 32, 1), (8, 3001, 1, 4, 33, 1)]


@pytest.mark.parametrize("B,L,n_min,n_max,K,min_hits", SHAPES,
                         ids=[f"B{s[0]}L{s[1]}n{s[2]}-{s[3]}K{s[4]}h{s[5]}" for s in SHAPES])
def test_parity_repetitive_contexts(B, L, n_min, n_max, K, min_hits):
    w = NgramWorkload("t", B=B, L=L, n_min=n_min, n_max=n_max, min_hits=min_hits, K=K)
    tokens, lengths = make_contexts(w, device="cuda", seed=B * 131 + L)
    c = _check(tokens, lengths, n_min, n_max, K, min_hits)
    if K > 0 and B >= 8:
        assert (c > 0).any()   # the contexts repeat: some drafts exist


@pytest.mark.parametrize("alphabet,B,L,n_max,min_hits", [(2, 64, 777, 12, 1), (3, 32, 5000, 6, 4),
                                                          (5, 128, 1003, 4, 1), (1, 16, 999, 8, 2),
                                                          (2, 40, 3001, 12, 3), (2, 24, 6000, 20, 7)])
def test_parity_small_alphabets(alphabet, B, L, n_max, min_hits):
    g = torch.Generator(device="cuda").manual_seed(alphabet * 17 + L)
    tokens = torch.randint(0, alphabet, (B, L), generator=g, device="cuda", dtype=torch.int32)
    lengths = torch.randint(0, L + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
    lengths[:4] = torch.tensor([0, 1, 2, L], dtype=torch.int32)
    _check(tokens, lengths, 1, n_max, 7, min_hits)


def test_unaligned_rows_take_the_scalar_loads():
    w = NgramWorkload("t", B=9, L=3001, n_min=1, n_max=5, min_hits=1, K=5)
    base, lengths = make_contexts(w, device="cuda", B=9, L=3002, seed=5)
    flat = base.reshape(-1)[1:1 + 9 * 3001]           # data pointer 4 bytes past a 16-byte boundary
    tokens = flat.view(9, 3001)
    assert tokens.data_ptr() % 16 != 0
    _check(tokens, lengths.clamp(max=3001), 1, 5, 5)
    aligned = base[:, :3000].contiguous()              # L % 4 == 0, aligned: vector loads
    _check(aligned, lengths.clamp(max=3000), 1, 5, 5)


def test_page_example_on_the_gpu():
    fields = {}
    for line in open(os.path.join(HERE, "golden", "glukhov_ngram_example.txt"), encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        fields[key] = vals
    words = fields["context"]
    vocab = {wd: i for i, wd in enumerate(sorted(set(words + fields["proposal"])))}
    t = torch.tensor([[vocab[wd] for wd in words]], dtype=torch.int32, device="cuda")
    K = int(fields["K"][0])
    draft, count = binding.spec_ngram_propose(t, torch.tensor([t.shape[1]], dtype=torch.int32, device="cuda"),
                                              int(fields["n_min"][0]), int(fields["n_max"][0]), K)
    inv = {i: wd for wd, i in vocab.items()}
    assert int(count[0]) == K
    assert [inv[int(v)] for v in draft[0].cpu()] == fields["proposal"]


def test_batch_sizes():
    """The launch picks about 6*SMs/B CTAs per sequence, each with at least
    4096 positions: from hundreds of CTAs per sequence (B = 1) to one."""
    for B in (1, 2, 5, 9, 19, 38, 76, 152, 1024):
        w = NgramWorkload("t", B=B, L=40000 if B < 200 else 8192, n_min=1, n_max=4, min_hits=1, K=5)
        tokens, lengths = make_contexts(w, device="cuda", seed=B)
        _check(tokens, lengths, 1, 4, 5)


@pytest.mark.parametrize("ctas", [1, 3, 8, 9, 37, 600])
def test_forced_ctas_per_sequence(ctas, monkeypatch):
    """Every mode combines its per-CTA partials the same way whatever the
    number of CTAs per sequence (SPEC_NGRAM_CTAS overrides the choice): up to
    8 through one cluster's shared memory, beyond that through global
    memory and the last CTA to finish."""
    monkeypatch.setenv("SPEC_NGRAM_CTAS", str(ctas))
    w = NgramWorkload("t", B=7, L=20000, n_min=1, n_max=4, min_hits=1, K=5)
    tokens, lengths = make_contexts(w, device="cuda", seed=ctas)
    for n_min, n_max, min_hits in ((1, 4, 1), (1, 6, 2), (1, 12, 3)):
        _check(tokens, lengths, n_min, n_max, 5, min_hits)


def test_runs_of_one_token():
    """Every position matches the suffix to n_max: all hits in one histogram bin."""
    tokens = torch.full((4, 9000), 7, dtype=torch.int32, device="cuda")
    lengths = torch.tensor([9000, 5, 1, 4096], dtype=torch.int32, device="cuda")
    c = _check(tokens, lengths, 1, 16, 5, min_hits=3)
    assert c.tolist() == [1, 1, 0, 1]


def test_invalid_length_marks_the_row():
    tokens = torch.zeros((3, 50), dtype=torch.int32, device="cuda")
    lengths = torch.tensor([10, 51, -1], dtype=torch.int32, device="cuda")
    draft, count = binding.spec_ngram_propose(tokens, lengths, 1, 4, 5)
    assert binding.spec_get_status() == 1                  # SPEC_ERR_ARG
    assert count.cpu().tolist() == [1, -1, -1]
    assert (draft[1:] == -1).all()
    assert binding.spec_get_status() == 0                  # cleared


def test_deterministic():
    w = NGRAM_WORKLOADS["ng1"]
    tokens, lengths = make_contexts(w, device="cuda")
    a = binding.spec_ngram_propose(tokens, lengths, w.n_min, w.n_max, w.K)
    b = binding.spec_ngram_propose(tokens, lengths, w.n_min, w.n_max, w.K)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("name", sorted(NGRAM_WORKLOADS))
def test_drafting_workload_full_size(name):
    w = NGRAM_WORKLOADS[name]
    tokens, lengths = make_contexts(w, device="cuda")
    _check(tokens, lengths, w.n_min, w.n_max, w.K, w.min_hits)
