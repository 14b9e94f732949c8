"""The no-allocation entry point (spec_verify_noalloc) gives the same outputs
as spec_verify.

It exists for callers that cannot allocate device memory while they run (an
engine whose memory pool owns nearly all of HBM, or a latency-critical loop
that cannot pay for cudaMalloc/cudaFree).  The tests call it through the C
ABI and compare every output with spec_verify's bit for bit (both run the same
kernels on the same bytes): two sampling calls in a row on different inputs,
a greedy (T = 0) call, and a call with a draft token out of range, whose
sequence is marked -1 as documented.  The array's status word is read back with
spec_noalloc_get_status, and a recorded timeout (set through the test hook,
no GPU stall involved) makes the next call's outputs -1 until it is read.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import Workload, make_chain

pytestmark = pytest.mark.gpu

SPEC_OK, SPEC_ERR_TOKEN_RANGE, SPEC_ERR_TIMEOUT = 0, 4, 6


def _noalloc(lib, zt, zd, x, T, seed):
    B, K1, V = zt.shape
    out = torch.full((B, K1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    vp = ctypes.c_void_p
    st = lib.spec_verify_noalloc(vp(zt.data_ptr()), vp(zd.data_ptr()) if zd is not None else None,
                                 vp(x.data_ptr()), B, K1 - 1, V, 0 if zt.dtype == torch.float32 else 1,
                                 ctypes.c_float(T), ctypes.c_uint64(seed), vp(out.data_ptr()),
                                 vp(n.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    return st, out, n


def _status(lib):
    return lib.spec_noalloc_get_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _same_as_spec_verify(lib, zt, zd, x, T, seed):
    ref_tok, ref_n = binding.spec_verify(zt, zd if T > 0 else None, x, T, seed)
    st, out, n = _noalloc(lib, zt, zd if T > 0 else None, x, T, seed)
    assert st == 0, lib.spec_last_error_message()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref_tok.cpu().numpy())
    assert np.array_equal(n.cpu().numpy(), ref_n.cpu().numpy())
    return out.cpu().numpy(), n.cpu().numpy()


def test_noalloc_matches_spec_verify_on_two_calls():
    lib = binding.library()
    assert _status(lib) == SPEC_OK
    cases = [
        (Workload("a", "chain", B=64, K=5, V=128256, dtype="bf16", T=0.7, sigma_t=3.0, sigma_d=0.5,
                  data_seed=11), 5),
        (Workload("b", "chain", B=24, K=3, V=32000, dtype="f32", T=1.0, sigma_t=3.0, sigma_d=1.0,
                  data_seed=12), 2 ** 40 + 9),
    ]
    for w, seed in cases:            # two calls in a row on the shared scratch
        zt, zd, x = make_chain(w, device="cuda")
        _same_as_spec_verify(lib, zt, zd, x, w.T, seed)
    assert _status(lib) == SPEC_OK


def test_noalloc_greedy_matches_spec_verify_and_the_oracle():
    lib = binding.library()
    w = Workload("g", "chain", B=16, K=4, V=50257, dtype="bf16", T=0.0, data_seed=14)
    zt, zd, x = make_chain(w, device="cuda")
    x[::2, 1] = zt[::2, 1].float().argmax(-1).to(torch.int32)   # some longer accepted prefixes
    out, n = _same_as_spec_verify(lib, zt, zd, x, 0.0, 0)
    ref = oracle.verify_chain(zt.cpu(), None, x.cpu(), 0.0, 0)
    assert np.array_equal(n, ref["n_accepted"]) and np.array_equal(out, ref["tokens"])
    assert _status(lib) == SPEC_OK


@pytest.mark.parametrize("T", [0.8, 0.0])
def test_noalloc_marks_a_draft_token_out_of_range(T):
    lib = binding.library()
    w = Workload("r", "chain", B=8, K=3, V=4096, dtype="f32", T=T, data_seed=15)
    zt, zd, x = make_chain(w, device="cuda")
    x[2, 1] = w.V                     # out of range: sequence 2 is marked -1
    x[5, 0] = -3
    out, n = _same_as_spec_verify(lib, zt, zd, x, T, 21)
    assert binding.spec_get_status() == SPEC_ERR_TOKEN_RANGE   # spec_verify's own word
    assert n[2] == -1 and n[5] == -1 and np.all(out[[2, 5]] == -1)
    assert _status(lib) == SPEC_ERR_TOKEN_RANGE                # the array's word, then cleared
    assert _status(lib) == SPEC_OK
    ref = oracle.verify_chain(zt.cpu(), zd.cpu() if T > 0 else None, x.cpu(), T, 21)
    assert np.array_equal(n == -1, ref["n_accepted"] == -1)


def test_noalloc_outputs_minus_one_after_an_unread_timeout():
    lib = binding.library()
    w = Workload("t", "chain", B=12, K=4, V=8192, dtype="bf16", T=1.0, data_seed=16)
    zt, zd, x = make_chain(w, device="cuda")
    assert _status(lib) == SPEC_OK
    assert lib.spec_debug_noalloc_status(4) == 0                # as a wait that ran out would
    st, out, n = _noalloc(lib, zt, zd, x, w.T, 3)
    assert st == 0
    torch.cuda.synchronize()
    assert np.all(n.cpu().numpy() == -1) and np.all(out.cpu().numpy() == -1)
    assert _status(lib) == SPEC_ERR_TIMEOUT
    _same_as_spec_verify(lib, zt, zd, x, w.T, 3)                # cleared: normal again
    assert _status(lib) == SPEC_OK


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = binding.library()
    lib.spec_verify_noalloc.restype = ctypes.c_int
    # 512 sequences x 5 rows x 63 slices of a 256000-entry fp32 row exceed the scratch
    vp = ctypes.c_void_p(256)
    st = lib.spec_verify_noalloc(vp, vp, vp, 512, 4, 256000, 0, ctypes.c_float(1.0),
                                 ctypes.c_uint64(0), vp, vp, None)
    assert st == 1
    assert b"scratch" in lib.spec_last_error_message()
