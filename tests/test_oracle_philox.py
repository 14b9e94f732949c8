"""Pins of the oracle's counter-based generator (Philox4x32-10) and uniforms.

Pinned against (1) the published known-answer vectors of Salmon et al.
(SC'11), stored in tests/golden/philox4x32_10_kat.txt, and (2) cuRAND's
host-side Philox4_32_10 generator, a library implementation run on the CPU:
its output block k for seed s is Philox(counter=(0, 0, k, 0), key=s).
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([int(w, 16) for w in line.split()])
    return rows


def test_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for r in rows:
        assert oracle.philox4x32_10(r[0:4], r[4:6]) == r[6:10]


def _curand():
    for name in ("libcurand.so.10", "libcurand.so", ctypes.util.find_library("curand")):
        if not name:
            continue
        for d in ("", "/usr/local/cuda/lib64/"):
            try:
                return ctypes.CDLL(d + name)
            except OSError:
                pass
    return None


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_matches_curand_host_generator(seed):
    lib = _curand()
    if lib is None:
        pytest.skip("cuRAND not available")
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        pytest.skip("cuRAND host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        nblk = 4096
        out = np.zeros(4 * nblk, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(out.size)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for k in list(range(64)) + list(range(nblk - 64, nblk)) + [777, 2048, 3001]:
        assert oracle.philox4x32_10([0, 0, k, 0], key) == [int(v) for v in out[4 * k:4 * k + 4]], k


def test_uniform_grid_and_range():
    us = np.array([oracle.uniform(12345, b, p, s) for b in range(64) for p in range(4)
                   for s in range(2)])
    assert np.all(us >= 0.0) and np.all(us <= 1.0 - 2.0 ** -24)
    k = us * 2 ** 24
    assert np.all(k == np.floor(k)), "u must lie on the 2^-24 grid"


def test_uniform_uses_word0_top_24_bits():
    # u(seed, b, position, slot) is fixed by the KAT-pinned block function:
    # the top 24 bits of word 0 of the block keyed (seed lo, seed hi) at
    # counter (b, position, slot, 0).
    seed = 0xA4093822299F31D0
    for (b, p, s) in [(0, 0, 0), (3, 1, 1), (65535, 7, 2), (2 ** 31, 2 ** 20, 1)]:
        w0 = oracle.philox4x32_10([b, p, s, 0], [seed & 0xFFFFFFFF, seed >> 32])[0]
        assert oracle.uniform(seed, b, p, s) == (w0 >> 8) / 2.0 ** 24


def test_uniform_is_uniform_and_slots_independent():
    n = 40000
    u0 = np.array([oracle.uniform(7, b, 3, 0) for b in range(n)])
    u1 = np.array([oracle.uniform(7, b, 3, 1) for b in range(n)])
    for u in (u0, u1):
        h, _ = np.histogram(u, bins=64, range=(0, 1))
        assert stats.chisquare(h).pvalue > 1e-3
    # slots 0 and 1 of the same (b, position) are uncorrelated
    r = np.corrcoef(u0, u1)[0, 1]
    assert abs(r) < 5.0 / np.sqrt(n)
