"""The bounded waits end: a kernel waiting on a barrier that nothing
completes gives up after its limit, the library reports SPEC_ERR_TIMEOUT,
and the stream and context stay usable (a verification call right after
matches the oracle)."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare_chain
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import Workload, make_chain

pytestmark = pytest.mark.gpu


def test_a_wait_that_never_completes_times_out():
    assert binding.spec_get_status() == 0
    t0 = time.perf_counter()
    assert binding.spec_selftest_wait() == 6                   # SPEC_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    # the wait gives up at 1 s of global time or after 2^17 polls, whichever
    # comes first; a poll suspends for at most 20 us and may wake sooner, so the
    # floor only shows that the kernel did wait
    assert 0.02 < waited < 30.0
    assert binding.spec_get_status() == 0                      # read once, then cleared
    w = Workload("after", "chain", B=8, K=4, V=4096, dtype="f32", T=1.0, data_seed=17)
    zt, zd, x = make_chain(w, device="cuda")
    out, n = binding.spec_verify(zt, zd, x, 1.0, 5)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_chain(zt.cpu(), zd.cpu(), x.cpu(), 1.0, 5)
    compare_chain(out.cpu().numpy(), n.cpu().numpy(), ref, positions=w.B * w.K)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_calls_after_an_unread_timeout_output_minus_one(T):
    """While a timeout is recorded and not yet read, a verification on the stream
    writes -1 (its statistics may be incomplete); reading the status clears it
    and the next call matches the oracle again."""
    lib = binding.library()
    assert binding.spec_get_status() == 0
    w = Workload("poison", "chain", B=6, K=3, V=2048, dtype="bf16", T=T, data_seed=23)
    zt, zd, x = make_chain(w, device="cuda")
    stream = torch.cuda.current_stream()
    assert lib.spec_selftest_wait(ctypes.c_void_p(stream.cuda_stream)) == 0   # records a timeout
    out, n = binding.spec_verify(zt, zd if T > 0 else None, x, T, 3)
    torch.cuda.synchronize()
    assert np.all(n.cpu().numpy() == -1) and np.all(out.cpu().numpy() == -1)
    assert binding.spec_get_status() == 6                      # SPEC_ERR_TIMEOUT, now cleared
    out, n = binding.spec_verify(zt, zd if T > 0 else None, x, T, 3)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_chain(zt.cpu(), zd.cpu() if T > 0 else None, x.cpu(), T, 3)
    if T > 0:
        compare_chain(out.cpu().numpy(), n.cpu().numpy(), ref, positions=w.B * w.K)
    else:
        assert np.array_equal(n.cpu().numpy(), ref["n_accepted"])
        assert np.array_equal(out.cpu().numpy(), ref["tokens"])
