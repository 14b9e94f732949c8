"""The no-allocation entry point (spec_verify_noalloc) gives the same outputs
as spec_verify.

It exists for callers that cannot allocate device memory while they run (an
engine whose memory pool owns nearly all of HBM, or a latency-critical loop
that cannot pay for cudaMalloc/cudaFree).  The test calls it through the C ABI
twice in a row, on different inputs, and compares every output with
spec_verify's bit for bit (both run the same kernels on the same bytes).  This
file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from sampling_row_online_gb300 import binding
from sampling_row_online_gb300.workloads import Workload, make_chain

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_spec_verify_on_two_calls():
    lib = binding.library()
    lib.spec_verify_noalloc.restype = ctypes.c_int
    cases = [
        (Workload("a", "chain", B=64, K=5, V=128256, dtype="bf16", T=0.7, sigma_t=3.0, sigma_d=0.5,
                  data_seed=11), 5),
        (Workload("b", "chain", B=24, K=3, V=32000, dtype="f32", T=1.0, sigma_t=3.0, sigma_d=1.0,
                  data_seed=12), 2 ** 40 + 9),
    ]
    for w, seed in cases:            # two calls in a row on the shared scratch
        zt, zd, x = make_chain(w, device="cuda")
        ref_tok, ref_n = binding.spec_verify(zt, zd, x, w.T, seed)
        st, out, n = _noalloc(lib, zt, zd, x, w.T, seed)
        assert st == 0, lib.spec_last_error_message()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref_tok.cpu().numpy())
        assert np.array_equal(n.cpu().numpy(), ref_n.cpu().numpy())


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = binding.library()
    lib.spec_verify_noalloc.restype = ctypes.c_int
    # 512 sequences x 5 rows x 63 slices of a 256000-entry fp32 row exceed the scratch
    vp = ctypes.c_void_p(256)
    st = lib.spec_verify_noalloc(vp, vp, vp, 512, 4, 256000, 0, ctypes.c_float(1.0),
                                 ctypes.c_uint64(0), vp, vp, None)
    assert st == 1
    assert b"scratch" in lib.spec_last_error_message()
