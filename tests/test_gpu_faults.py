"""Host-side fault injection (no GPU fault involved): a launch made to fail
through the library's launch hook returns SPEC_ERR_CUDA, and the next call on
the same stream is correct: the first launch of a call failing leaves the
workspace untouched; the second (decision) launch failing after the
streaming kernel ran puts the item tickets back to zero."""
import numpy as np
import pytest

import oracle
from gpu_helpers import compare_chain
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import NgramWorkload, Workload, make_chain, make_contexts

pytestmark = pytest.mark.gpu


def _chain_ok(seed):
    w = Workload("f", "chain", B=16, K=5, V=32000, dtype="bf16", T=0.7, data_seed=seed)
    zt, zd, x = make_chain(w, device="cuda")
    out, n = binding.spec_verify(zt, zd, x, w.T, 3)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_chain(zt.cpu(), zd.cpu(), x.cpu(), w.T, 3)
    compare_chain(out.cpu().numpy(), n.cpu().numpy(), ref, positions=w.B * w.K)
    return zt, zd, x


@pytest.mark.parametrize("nth", [1, 2])
def test_failed_launch_then_a_correct_call(nth):
    lib = binding.library()
    zt, zd, x = _chain_ok(61)
    assert lib.spec_debug_fail_launch(nth) == 0
    with pytest.raises(binding.SpecError) as e:
        binding.spec_verify(zt, zd, x, 0.7, 3)
    assert e.value.status == 5                                   # SPEC_ERR_CUDA
    assert binding.spec_get_status() == 0
    for seed in (62, 63):
        _chain_ok(seed)


def test_failed_drafter_and_tree_launches():
    lib = binding.library()
    w = NgramWorkload("f", B=8, L=4000, n_min=1, n_max=4, min_hits=1, K=5, data_seed=7)
    tokens, lengths = make_contexts(w, device="cuda")
    assert lib.spec_debug_fail_launch(1) == 0
    with pytest.raises(binding.SpecError):
        binding.spec_ngram_propose(tokens, lengths, 1, 4, 5)
    draft, count = binding.spec_ngram_propose(tokens, lengths, 1, 4, 5)   # the counters were not touched
    assert binding.spec_get_status() == 0
    rd, rc = oracle.ngram_propose(tokens.cpu().numpy(), lengths.cpu().numpy(), 1, 4, 5)
    assert np.array_equal(count.cpu().numpy(), rc) and np.array_equal(draft.cpu().numpy(), rd)
    import torch
    assert lib.spec_debug_fail_launch(1) == 0
    with pytest.raises(binding.SpecError):
        binding.spec_tree_mask(torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32, device="cuda"))
    assert lib.spec_debug_fail_launch(0) == 0
