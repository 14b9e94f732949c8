"""The binding's thin wrappers that other tests do not reach directly: the
no-allocation chain call, the per-sequence tree calls, and the measurement
hook.  Each must give exactly what the call it stands beside gives."""
import pytest
import torch

from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import Workload, make_chain, make_tree

pytestmark = pytest.mark.gpu


def test_noalloc_equals_spec_verify():
    w = Workload("w", "chain", B=24, K=4, V=32000, dtype="bf16", T=0.9, data_seed=71)
    zt, zd, x = make_chain(w, device="cuda")
    a = binding.spec_verify_noalloc(zt, zd, x, w.T, 5)
    b = binding.spec_verify(zt, zd, x, w.T, 5)
    assert binding.spec_get_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_per_sequence_tree_wrappers_equal_the_two_dimensional_parent_form():
    w = Workload("w", "tree", B=6, K=63, V=4096, dtype="bf16", T=0.0, data_seed=72)
    zt, parent, tok = make_tree(w, device="cuda")
    pars = parent.unsqueeze(0).expand(w.B, -1).contiguous()
    a = binding.spec_verify_trees_greedy(zt, pars, tok)
    b = binding.spec_verify_tree_greedy(zt, parent, tok)
    assert binding.spec_get_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    with pytest.raises(ValueError):
        binding.spec_verify_trees_greedy(zt, parent, tok)
    zd = (torch.randn(zt.shape, device="cuda") * 2).to(zt.dtype)
    c = binding.spec_verify_trees(zt, zd, pars, tok, 0.8, 9)
    d = binding.spec_verify_tree(zt, zd, parent, tok, 0.8, 9)
    assert binding.spec_get_status() == 0
    assert torch.equal(c[0], d[0]) and torch.equal(c[1], d[1])


def test_rows_event_hook_brackets_the_streaming_kernel():
    w = Workload("w", "chain", B=16, K=5, V=128256, dtype="bf16", T=0.7, data_seed=73)
    zt, zd, x = make_chain(w, device="cuda")
    ref = binding.spec_verify(zt, zd, x, w.T, 2)
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    for e in (e0, e1, e2):
        e.record()
    torch.cuda.synchronize()
    e0.record()
    binding.spec_arm_rows_event(e1)
    out = binding.spec_verify(zt, zd, x, w.T, 2)
    e2.record()
    torch.cuda.synchronize()
    assert binding.spec_get_status() == 0
    assert torch.equal(out[0], ref[0]) and torch.equal(out[1], ref[1])
    rows, total = e0.elapsed_time(e1), e0.elapsed_time(e2)
    assert 0.0 < rows <= total


def test_error_strings():
    assert binding.spec_error_string(0) == "SPEC_OK"
    assert binding.spec_error_string(6) == "SPEC_ERR_TIMEOUT"
    binding.spec_debug_fail_launch(0)
