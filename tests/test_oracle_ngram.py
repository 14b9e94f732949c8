"""Pins of the oracle's n-gram (prompt-lookup) drafter: the page's worked
example (a golden fixture), a hand case of min_hits, and on random repetitive
contexts an independent check of its defining properties with byte-string
search: the proposal follows an earlier occurrence of the longest suffix
(n <= n_max) seen at least min_hits times before, that occurrence is the most
recent one, and nothing is proposed only when no suffix of length >= n_min
was seen min_hits times."""
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    fields = {}
    for line in open(os.path.join(HERE, "golden", "glukhov_ngram_example.txt"), encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        fields[key] = vals
    return fields


def test_page_example():
    f = _golden()
    words = f["context"]
    vocab = {w: i for i, w in enumerate(sorted(set(words + f["proposal"])))}
    t = np.array([vocab[w] for w in words], dtype=np.int32)
    K = int(f["K"][0])
    draft, count = oracle.ngram_propose(t[None], [len(t)], int(f["n_min"][0]), int(f["n_max"][0]), K)
    inv = {i: w for w, i in vocab.items()}
    assert count[0] == K
    assert [inv[int(v)] for v in draft[0]] == f["proposal"]


def _enc(a):
    return np.asarray(a, dtype="<i4").tobytes()


def _occurrences(t, n, end_limit):
    """Every start j with t[j:j+n] == t[-n:] and j + n <= end_limit, found with
    bytes.rfind on the 4-byte token encoding (hits across token boundaries
    are skipped)."""
    hay = _enc(t[:end_limit])
    needle = _enc(t[len(t) - n:])
    out = []
    hi = len(hay)
    while True:
        pos = hay.rfind(needle, 0, hi)
        if pos < 0:
            return out
        if pos % 4 == 0:
            out.append(pos // 4)
        hi = pos + len(needle) - 1  # the next candidate ends before this one does


@pytest.mark.parametrize("alphabet,L,n_min,n_max,K,min_hits", [(3, 60, 1, 4, 5, 1), (5, 200, 2, 6, 3, 1),
                                                               (20, 400, 1, 3, 8, 1), (2, 30, 1, 10, 2, 1),
                                                               (50, 1000, 3, 8, 4, 1), (3, 80, 1, 5, 4, 2),
                                                               (8, 300, 2, 6, 6, 3), (2, 40, 1, 12, 3, 5)])
def test_properties_on_random_contexts(alphabet, L, n_min, n_max, K, min_hits):
    rng = np.random.default_rng(alphabet * 7 + L + min_hits)
    B = 300
    tokens = rng.integers(0, alphabet, (B, L)).astype(np.int32)
    # repeats: copy earlier spans forward, as in code editing
    for b in range(0, B, 2):
        for _ in range(3):
            src = rng.integers(0, L // 2)
            n = rng.integers(2, 12)
            dst = rng.integers(src + 1, L)
            m = min(n, L - dst, dst - src)
            tokens[b, dst:dst + m] = tokens[b, src:src + m]
    lengths = rng.integers(0, L + 1, B).astype(np.int32)
    draft, count = oracle.ngram_propose(tokens, lengths, n_min, n_max, K, min_hits=min_hits)
    for b in range(B):
        ln = int(lengths[b])
        t = tokens[b, :ln]
        found = None
        for n in range(min(n_max, ln - 1), n_min - 1, -1):
            occ = _occurrences(t, n, ln - 1)
            if len(occ) >= min_hits:
                found = (n, max(occ))
                break
        if found is None:
            assert count[b] == 0 and np.all(draft[b] == -1)
            continue
        n, j = found
        c = min(K, ln - (j + n))
        assert count[b] == c
        assert np.array_equal(draft[b, :c], t[j + n:j + n + c])
        assert np.all(draft[b, c:] == -1)


def test_min_hits_hand_case():
    """p q c X a b c Y a b c: the suffix (a, b, c) and (b, c) were seen once
    before, (c) twice (after q and after b)."""
    p, q, a, b, c, X, Y = range(7)
    t = np.array([[p, q, c, X, a, b, c, Y, a, b, c]], dtype=np.int32)
    d, n = oracle.ngram_propose(t, [11], 1, 3, 3, min_hits=1)
    assert n[0] == 3 and d[0].tolist() == [Y, a, b]       # after (a, b, c) at j = 4
    d, n = oracle.ngram_propose(t, [11], 1, 3, 3, min_hits=2)
    assert n[0] == 3 and d[0].tolist() == [Y, a, b]       # (c): most recent at j = 6
    d, n = oracle.ngram_propose(t, [11], 2, 3, 3, min_hits=2)
    assert n[0] == 0 and d[0].tolist() == [-1, -1, -1]    # no n >= 2 seen twice
    d, n = oracle.ngram_propose(t, [11], 1, 3, 3, min_hits=3)
    assert n[0] == 0
    d, n = oracle.ngram_propose(t, [8], 1, 3, 5, min_hits=2)   # context p q c X a b c Y
    assert n[0] == 0                                           # (Y) never seen before


def test_edge_cases():
    t = np.array([[7, 7, 7, 7, 0, 0]], dtype=np.int32)
    # a run: the suffix (7, 7) of length 4's prefix occurs overlapping itself
    d, c = oracle.ngram_propose(t, [4], 1, 3, 2)
    assert c[0] == 1 and d[0].tolist() == [7, -1]
    d, c = oracle.ngram_propose(t, [1], 1, 3, 2)   # one token: nothing earlier
    assert c[0] == 0
    d, c = oracle.ngram_propose(t, [0], 1, 3, 2)   # empty context
    assert c[0] == 0
    d, c = oracle.ngram_propose(t, [6], 1, 3, 0)   # K = 0
    assert c[0] == 0 and d.shape == (1, 0)
    with pytest.raises(ValueError):
        oracle.ngram_propose(t, [6], 0, 3, 2)
    with pytest.raises(ValueError):
        oracle.ngram_propose(t, [6], 1, 3, 2, min_hits=0)
    with pytest.raises(ValueError):
        oracle.ngram_propose(t, [7], 1, 3, 2)
