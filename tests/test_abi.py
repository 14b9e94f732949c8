"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host before touching CUDA (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sampling_row_online_gb300 import build, binding
    build.build()
    return binding.library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("spec_verify", "spec_verify_tree_greedy", "spec_verify_tree", "spec_verify_ex", "spec_verify_host",
                     "spec_tree_max_depth", "spec_tree_mask", "spec_ngram_propose", "spec_topk",
                     "spec_eagle2_expand", "spec_eagle2_rerank", "spec_verify_trees_greedy",
                     "spec_verify_trees", "spec_verify_points", "spec_selftest_wait", "spec_debug_fail_launch", "spec_get_status",
                     "spec_error_string", "spec_last_error_message", "spec_shutdown"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_has_a_wrapper_of_the_same_name_for_every_declared_call():
    import sampling_row_online_gb300 as pkg
    from sampling_row_online_gb300 import binding
    for name in _declared_functions():
        assert callable(getattr(binding, name, None)), name
        assert name in pkg.__all__, name


def _verify(lib, **kw):
    a = dict(zt=ctypes.c_void_p(16), zd=ctypes.c_void_p(16), x=ctypes.c_void_p(16), B=2, K=3,
             V=100, dtype=1, T=1.0, seed=0, out=ctypes.c_void_p(16), n=ctypes.c_void_p(16),
             stream=None)
    a.update(kw)
    return lib.spec_verify(a["zt"], a["zd"], a["x"], a["B"], a["K"], a["V"], a["dtype"], a["T"],
                           a["seed"], a["out"], a["n"], a["stream"])


def test_argument_validation_without_gpu(lib):
    ARG, DTYPE = 1, 2
    assert _verify(lib, B=0) == 0                       # empty batch: no-op
    assert _verify(lib, B=-1) == ARG
    assert _verify(lib, V=0) == ARG
    assert _verify(lib, K=-1) == ARG
    assert _verify(lib, K=256) == ARG
    assert _verify(lib, dtype=7) == DTYPE
    assert _verify(lib, T=-0.5) == ARG
    assert _verify(lib, T=float("nan")) == ARG
    assert _verify(lib, T=float("inf")) == ARG
    assert _verify(lib, T=1e-40) == ARG                  # 1/T overflows fp32
    assert _verify(lib, zt=None) == ARG
    assert _verify(lib, zd=None) == ARG                  # T > 0 needs draft logits
    assert _verify(lib, x=None) == ARG
    assert _verify(lib, out=None) == ARG
    assert _verify(lib, n=None) == ARG
    msg = lib.spec_last_error_message().decode()
    assert "NULL" in msg
    assert lib.spec_error_string(ARG) == b"SPEC_ERR_ARG"
    assert lib.spec_error_string(0) == b"SPEC_OK"


def test_tree_validation_without_gpu(lib):
    vp = ctypes.c_void_p(16)
    assert lib.spec_verify_tree_greedy(vp, vp, vp, 2, 0, 10, 1, 0, vp, vp, None) == 1     # N = 0
    assert lib.spec_verify_tree_greedy(vp, vp, vp, 2, 5, 10, 1, 5, vp, vp, None) == 1     # depth >= N
    assert lib.spec_verify_tree_greedy(vp, vp, vp, 0, 5, 10, 1, 2, vp, vp, None) == 0     # empty
    assert lib.spec_tree_mask(vp, 1, 0, vp, vp, None) == 1
    # stochastic tree: (zt, zd, parent, tokens, B, N, V, dtype, T, seed, D, path, len, stream)
    t = lib.spec_verify_tree
    assert t(vp, vp, vp, vp, 2, 0, 10, 1, 1.0, 0, 0, vp, vp, None) == 1                  # N = 0
    assert t(vp, vp, vp, vp, 2, 5, 10, 1, 1.0, 0, 5, vp, vp, None) == 1                  # depth >= N
    assert t(vp, vp, vp, vp, 2, 5, 10, 1, -1.0, 0, 2, vp, vp, None) == 1                 # T < 0
    assert t(vp, None, vp, vp, 2, 5, 10, 1, 1.0, 0, 2, vp, vp, None) == 1                # no draft rows
    assert t(vp, vp, vp, vp, 2, 5, 10, 9, 1.0, 0, 2, vp, vp, None) == 2                  # dtype
    assert t(vp, vp, vp, vp, 0, 5, 10, 1, 1.0, 0, 2, vp, vp, None) == 0                  # empty


def test_ngram_validation_without_gpu(lib):
    vp = ctypes.c_void_p(16)
    g = lib.spec_ngram_propose   # (tokens, lengths, B, L, n_min, n_max, min_hits, K, draft, count, stream)
    assert g(vp, vp, 0, 10, 1, 4, 1, 5, vp, vp, None) == 0        # empty batch
    assert g(vp, vp, -1, 10, 1, 4, 1, 5, vp, vp, None) == 1       # B < 0
    assert g(vp, vp, 2, -1, 1, 4, 1, 5, vp, vp, None) == 1        # L < 0
    assert g(vp, vp, 2, 10, 0, 4, 1, 5, vp, vp, None) == 1        # n_min < 1
    assert g(vp, vp, 2, 10, 5, 4, 1, 5, vp, vp, None) == 1        # n_max < n_min
    assert g(vp, vp, 2, 10, 1, 65, 1, 5, vp, vp, None) == 1       # n_max > 64
    assert g(vp, vp, 2, 10, 1, 4, 0, 5, vp, vp, None) == 1        # min_hits < 1
    assert g(vp, vp, 2, 10, 1, 4, 1, 256, vp, vp, None) == 1      # K > 255
    assert g(vp, None, 2, 10, 1, 4, 1, 5, vp, vp, None) == 1      # no lengths
    assert g(vp, vp, 2, 10, 1, 4, 1, 5, None, vp, None) == 1      # no draft output with K > 0
    assert g(None, vp, 2, 10, 1, 4, 1, 5, vp, vp, None) == 1      # no tokens with L > 0


def test_eagle2_validation_without_gpu(lib):
    vp = ctypes.c_void_p(16)
    t = lib.spec_topk            # (logits, R, V, dtype, T, k, tokens, prob, stream)
    assert t(vp, 0, 100, 1, 1.0, 5, vp, vp, None) == 0            # no rows
    assert t(vp, 4, 100, 7, 1.0, 5, vp, vp, None) == 2            # dtype
    assert t(vp, 4, 100, 1, 1.0, 0, vp, vp, None) == 1            # k < 1
    assert t(vp, 4, 100, 1, 1.0, 33, vp, vp, None) == 1           # k > 32
    assert t(vp, 4, 3, 1, 1.0, 4, vp, vp, None) == 1              # k > V
    assert t(vp, 4, 100, 1, 0.0, 5, vp, vp, None) == 1            # T = 0
    assert t(None, 4, 100, 1, 1.0, 5, vp, vp, None) == 1          # NULL
    e = lib.spec_eagle2_expand   # (z, frontier, B, F, V, dtype, T, k, tok, val, par, cap, offset, k_next, next, stream)
    assert e(vp, vp, 0, 4, 100, 1, 1.0, 4, vp, vp, vp, 40, 1, 4, vp, None) == 0     # empty batch
    assert e(vp, vp, 2, 4, 100, 1, 1.0, 4, vp, vp, vp, 16, 1, 4, vp, None) == 1     # offset + F*k > cap
    assert e(vp, vp, 2, 4, 100, 1, 1.0, 4, vp, vp, vp, 40, 0, 4, vp, None) == 1     # offset < 1
    assert e(vp, vp, 2, 4, 100, 1, 1.0, 4, vp, vp, vp, 40, 1, 17, vp, None) == 1    # k_next > F*k
    assert e(vp, vp, 2, 200, 100, 1, 1.0, 32, vp, vp, vp, 9000, 1, 4, vp, None) == 1  # F*k > 4096
    r = lib.spec_eagle2_rerank   # (val, par, tok, B, M, m, par_out, tok_out, idx_out, stream)
    assert r(vp, vp, vp, 0, 10, 5, vp, vp, vp, None) == 0
    assert r(vp, vp, vp, 2, 10, 10, vp, vp, vp, None) == 1          # m > M - 1
    assert r(vp, vp, vp, 2, 9000, 5, vp, vp, vp, None) == 1         # M > 8192
    assert r(vp, vp, vp, 2, 10, 5, None, vp, vp, None) == 1


@pytest.mark.parametrize("parent,depth", [([-1], 0), ([-1, 0, 0, 1, 2], 2),
                                          ([-1, 0, 1, 2, 3], 4), ([-1, 0, 0, 0], 1)])
def test_tree_max_depth_host(lib, parent, depth):
    p = np.array(parent, dtype=np.int32)
    assert lib.spec_tree_max_depth(p.ctypes.data_as(ctypes.c_void_p), p.size) == depth


@pytest.mark.parametrize("parent", [[0], [-1, 1], [-1, 0, 3], [-1, -1]])
def test_tree_max_depth_rejects_non_trees(lib, parent):
    p = np.array(parent, dtype=np.int32)
    assert lib.spec_tree_max_depth(p.ctypes.data_as(ctypes.c_void_p), p.size) == -7


def test_binding_matches_oracle_tree_depth(lib):
    import oracle
    from sampling_row_online_gb300 import binding
    from sampling_row_online_gb300.workloads import tree_parents
    parent = tree_parents((4, 3, 2, 2, 1), 63)
    assert binding.spec_tree_max_depth(parent) == oracle.tree_max_depth(parent) == 4
