"""Reference oracle (fp64, CPU) for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``sampling_row_online_gb300``) never imports it, and the two share
no code.  The arithmetic lives in ``oracle.c`` (plain C, fp64, left-to-right
loops); this module only marshals arrays through ctypes.

Inputs are CPU tensors (``torch.float32`` / ``torch.bfloat16``) or numpy arrays
(``float32``; ``uint16``/``int16`` holding bfloat16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

F32, BF16 = 0, 1
OK, ERR_ARG, ERR_TOKEN, ERR_PARENT = 0, 1, 2, 3


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c_p = ctypes.c_void_p
        i32, u32, u64, f64 = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
        lib.oracle_philox4x32_10.argtypes = [c_p, c_p, c_p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_uniform.argtypes = [u64, u32, u32, u32]
        lib.oracle_uniform.restype = f64
        lib.oracle_row_stats.argtypes = [c_p, i32, i32, f64, c_p, c_p]
        lib.oracle_row_stats.restype = None
        lib.oracle_argmax.argtypes = [c_p, i32, i32]
        lib.oracle_argmax.restype = i32
        lib.oracle_accept.argtypes = [c_p, c_p, i32, i32, f64, i32, f64, c_p, c_p]
        lib.oracle_accept.restype = i32
        lib.oracle_target_sample.argtypes = [c_p, i32, i32, f64, f64, c_p]
        lib.oracle_target_sample.restype = i32
        lib.oracle_residual_sample.argtypes = [c_p, c_p, i32, i32, f64, f64, c_p, c_p]
        lib.oracle_residual_sample.restype = i32
        lib.oracle_verify_chain.argtypes = [c_p, c_p, c_p, i32, i32, i32, i32, f64, u64,
                                            c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, i32]
        lib.oracle_verify_chain.restype = i32
        lib.oracle_tree_max_depth.argtypes = [c_p, i32]
        lib.oracle_tree_max_depth.restype = i32
        lib.oracle_tree_mask.argtypes = [c_p, i32, c_p, c_p]
        lib.oracle_tree_mask.restype = i32
        lib.oracle_verify_tree_greedy.argtypes = [c_p, c_p, c_p, i32, i32, i32, i32, i32,
                                                  c_p, c_p, i32]
        lib.oracle_verify_tree_greedy.restype = i32
        lib.oracle_verify_tree_sample.argtypes = [c_p, c_p, c_p, c_p, i32, i32, i32, i32, f64,
                                                  u64, i32, c_p, c_p, c_p, c_p, c_p, c_p, c_p,
                                                  i32]
        lib.oracle_verify_tree_sample.restype = i32
        lib.oracle_ngram_propose.argtypes = [c_p, c_p, i32, i32, i32, i32, i32, i32, c_p, c_p]
        lib.oracle_ngram_propose.restype = i32
        lib.oracle_verify_points.argtypes = [c_p, c_p, c_p, i32, i32, i32, i32, ctypes.c_double, u64, c_p, c_p, c_p,
                                             c_p, i32]
        lib.oracle_verify_points.restype = i32
        lib.oracle_topk_prob.argtypes = [c_p, i32, i32, i32, ctypes.c_double, i32, c_p, c_p]
        lib.oracle_topk_prob.restype = i32
        lib.oracle_eagle2_expand.argtypes = [c_p, i32, i32, i32, c_p, c_p, c_p, c_p, c_p, i32, i32, i32, c_p, c_p]
        lib.oracle_eagle2_expand.restype = i32
        lib.oracle_eagle2_rerank.argtypes = [c_p, c_p, c_p, i32, i32, i32, c_p, c_p, c_p, c_p]
        lib.oracle_eagle2_rerank.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ----------------------------------------------------------------------------
# array marshalling
# ----------------------------------------------------------------------------
def _logits(z):
    """Return (contiguous numpy array holding the raw element bits, dtype code)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(z, torch.Tensor):
        z = z.detach()
        if z.device.type != "cpu":
            raise ValueError("oracle inputs must be CPU tensors")
        z = z.contiguous()
        if z.dtype == torch.float32:
            return z.numpy(), F32
        if z.dtype == torch.bfloat16:
            return z.view(torch.int16).numpy(), BF16
        raise TypeError(f"unsupported logits dtype {z.dtype}")
    a = np.ascontiguousarray(z)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype in (np.uint16, np.int16):
        return a, BF16
    if a.dtype == np.float64:
        raise TypeError("pass float32 (or bfloat16 bits); the oracle widens exactly itself")
    raise TypeError(f"unsupported logits dtype {a.dtype}")


def _i32(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# public helpers
# ----------------------------------------------------------------------------
def philox4x32_10(ctr, key):
    """Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return [int(v) for v in out]


def uniform(seed: int, b: int, position: int, slot: int) -> float:
    """u = (word0 >> 8) * 2^-24 of Philox(counter=(b, position, slot, 0), key=seed)."""
    return float(_load().oracle_uniform(seed, b, position, slot))


def row_stats(z, T: float):
    """(m, S) = (max z, sum exp((z - m) / T)) of one row, in fp64."""
    a, dt = _logits(z)
    m, S = ctypes.c_double(), ctypes.c_double()
    _load().oracle_row_stats(_ptr(a), dt, a.size, float(T), ctypes.byref(m), ctypes.byref(S))
    return m.value, S.value


def argmax(z) -> int:
    a, dt = _logits(z)
    return int(_load().oracle_argmax(_ptr(a), dt, a.size))


def accept(zt, zd, x: int, T: float, u: float):
    """(accepted, r = p(x)/q(x), near) for one draft token under uniform u."""
    a, dt = _logits(zt)
    d, dt2 = _logits(zd)
    assert dt == dt2 and a.size == d.size
    r, near = ctypes.c_double(), ctypes.c_int()
    ok = _load().oracle_accept(_ptr(a), _ptr(d), dt, a.size, float(T), int(x), float(u),
                               ctypes.byref(r), ctypes.byref(near))
    return bool(ok), r.value, bool(near.value)


def target_sample(zt, T: float, u: float):
    """(token, near) drawn from p = softmax(zt / T) by inverse CDF at uniform u."""
    a, dt = _logits(zt)
    near = ctypes.c_int()
    tok = _load().oracle_target_sample(_ptr(a), dt, a.size, float(T), float(u), ctypes.byref(near))
    return int(tok), bool(near.value)


def residual_sample(zt, zd, T: float, u: float):
    """(token, near, fallback) drawn from norm(max(0, p - q)) at uniform u."""
    a, dt = _logits(zt)
    d, _ = _logits(zd)
    near, fb = ctypes.c_int(), ctypes.c_int()
    tok = _load().oracle_residual_sample(_ptr(a), _ptr(d), dt, a.size, float(T), float(u),
                                         ctypes.byref(near), ctypes.byref(fb))
    return int(tok), bool(near.value), bool(fb.value)


def verify_chain(zt, zd, draft_tokens, T: float, seed: int, *, b_ids=None, u_acc=None,
                 u_samp=None, want_stats=False, nthreads=1):
    """Chain verification of nb sequences.

    zt: [nb, K+1, V]; zd: [nb, K, V] (may be None when T == 0); draft_tokens: [nb, K].
    Returns a dict with tokens [nb, K+1], n_accepted [nb], near [nb], fallback [nb],
    status, and (want_stats) row_max / row_sumexp [nb, 2K+1].
    """
    zt_a, dt = _logits(zt)
    nb, K1, V = zt_a.shape
    K = K1 - 1
    zd_a = None
    if zd is not None and K > 0:
        zd_a, dt2 = _logits(zd)
        assert dt2 == dt and zd_a.shape == (nb, K, V)
    elif T > 0 and K > 0:
        raise ValueError("draft logits are required when T > 0")
    x = _i32(draft_tokens).reshape(nb, K)
    bi = None if b_ids is None else _i32(b_ids).reshape(nb)
    ua = None if u_acc is None else np.ascontiguousarray(u_acc, dtype=np.float64).reshape(nb, K)
    us = None if u_samp is None else np.ascontiguousarray(u_samp, dtype=np.float64).reshape(nb, K + 1)
    tokens = np.zeros((nb, K + 1), dtype=np.int32)
    n = np.zeros(nb, dtype=np.int32)
    near = np.zeros(nb, dtype=np.int32)
    fb = np.zeros(nb, dtype=np.int32)
    m = S = None
    if want_stats:
        m = np.zeros((nb, 2 * K + 1), dtype=np.float64)
        S = np.zeros((nb, 2 * K + 1), dtype=np.float64)
    st = _load().oracle_verify_chain(_ptr(zt_a), _ptr(zd_a), _ptr(x), nb, K, V, dt, float(T),
                                     int(seed) & ((1 << 64) - 1), _ptr(bi), _ptr(ua), _ptr(us),
                                     _ptr(tokens), _ptr(n), _ptr(near), _ptr(fb), _ptr(m),
                                     _ptr(S), int(nthreads))
    if st == ERR_ARG:
        raise ValueError("oracle_verify_chain: invalid arguments")
    out = dict(tokens=tokens, n_accepted=n, near=near.astype(bool), fallback=fb.astype(bool),
               status=st)
    if want_stats:
        out["row_max"] = m
        out["row_sumexp"] = S
    return out


def tree_max_depth(parent) -> int:
    p = _i32(parent)
    return int(_load().oracle_tree_max_depth(_ptr(p), p.size))


def tree_mask(parent):
    """(mask [N, N] uint8, depth [N]) of the tree given by parent[]."""
    p = _i32(parent)
    N = p.size
    mask = np.zeros((N, N), dtype=np.uint8)
    depth = np.zeros(N, dtype=np.int32)
    st = _load().oracle_tree_mask(_ptr(p), N, _ptr(mask), _ptr(depth))
    if st != OK:
        raise ValueError("invalid parent array")
    return mask, depth


def verify_tree_greedy(zt, parent, node_tokens, *, max_depth=None, nthreads=1):
    """Greedy tree verification; returns (path [nb, D+1], length [nb], status)."""
    zt_a, dt = _logits(zt)
    nb, N, V = zt_a.shape
    p = _i32(parent).reshape(N)
    tok = _i32(node_tokens).reshape(nb, N)
    D = tree_max_depth(p) if max_depth is None else int(max_depth)
    if D < 0:
        raise ValueError("invalid parent array")
    path = np.zeros((nb, D + 1), dtype=np.int32)
    length = np.zeros(nb, dtype=np.int32)
    st = _load().oracle_verify_tree_greedy(_ptr(zt_a), _ptr(p), _ptr(tok), nb, N, V, dt, D,
                                           _ptr(path), _ptr(length), int(nthreads))
    if st in (ERR_ARG, ERR_PARENT):
        raise ValueError("oracle_verify_tree_greedy: invalid arguments")
    return path, length, st


def verify_tree_sample(zt, zd, parent, node_tokens, T: float, seed: int, *, max_depth=None,
                       b_ids=None, u_acc=None, u_samp=None, nthreads=1):
    """Stochastic tree verification (candidates tried sibling by sibling with
    the residual updated after each reject).

    zt, zd: [nb, N, V]; parent: [N]; node_tokens: [nb, N]; u_acc / u_samp: optional
    [nb, N] uniforms (test of child c / draw at node u).  Returns a dict with
    path [nb, D+1], length [nb], near [nb], fallback [nb], status.
    """
    zt_a, dt = _logits(zt)
    zd_a, dt2 = _logits(zd)
    nb, N, V = zt_a.shape
    assert dt2 == dt and zd_a.shape == (nb, N, V)
    p = _i32(parent).reshape(N)
    tok = _i32(node_tokens).reshape(nb, N)
    D = tree_max_depth(p) if max_depth is None else int(max_depth)
    if D < 0:
        raise ValueError("invalid parent array")
    bi = None if b_ids is None else _i32(b_ids).reshape(nb)
    ua = None if u_acc is None else np.ascontiguousarray(u_acc, dtype=np.float64).reshape(nb, N)
    us = None if u_samp is None else np.ascontiguousarray(u_samp, dtype=np.float64).reshape(nb, N)
    path = np.zeros((nb, D + 1), dtype=np.int32)
    length = np.zeros(nb, dtype=np.int32)
    near = np.zeros(nb, dtype=np.int32)
    fb = np.zeros(nb, dtype=np.int32)
    st = _load().oracle_verify_tree_sample(_ptr(zt_a), _ptr(zd_a), _ptr(p), _ptr(tok), nb, N, V,
                                           dt, float(T), int(seed) & ((1 << 64) - 1), D,
                                           _ptr(bi), _ptr(ua), _ptr(us), _ptr(path),
                                           _ptr(length), _ptr(near), _ptr(fb), int(nthreads))
    if st in (ERR_ARG, ERR_PARENT):
        raise ValueError("oracle_verify_tree_sample: invalid arguments")
    return dict(path=path, length=length, near=near.astype(bool), fallback=fb.astype(bool),
                status=st)


def ngram_propose(tokens, lengths, n_min: int, n_max: int, K: int, min_hits: int = 1):
    """n-gram (prompt-lookup) proposals: (draft [B, K] int32, -1 padded; count [B])."""
    t = _i32(tokens)
    if t.ndim == 1:
        t = t.reshape(1, -1)
    B, L = t.shape
    ln = _i32(lengths).reshape(B)
    draft = np.zeros((B, K), dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    st = _load().oracle_ngram_propose(_ptr(t), _ptr(ln), B, L, int(n_min), int(n_max), int(min_hits),
                                      int(K), _ptr(draft), _ptr(count))
    if st != OK:
        raise ValueError("oracle_ngram_propose: invalid arguments")
    return draft, count


def topk_prob(z, k: int, T: float = 1.0):
    """Per row of z [R, V] (or [..., V]): the k tokens of largest logit (ties:
    lower index first) and their probabilities under softmax(z / T).
    Returns (tokens [R, k] int32, prob [R, k] float64)."""
    a, dt = _logits(z)
    V = a.shape[-1]
    R = int(a.size // V) if V else 0
    tok = np.zeros((R, k), dtype=np.int32)
    prob = np.zeros((R, k), dtype=np.float64)
    st = _load().oracle_topk_prob(_ptr(a), R, V, dt, float(T), int(k), _ptr(tok), _ptr(prob))
    if st != OK:
        raise ValueError("oracle_topk_prob: invalid arguments")
    return tok, prob


def eagle2_expand(frontier, topk_tok, topk_prob_, node_tok, node_val, node_par, offset: int, k_next: int):
    """One expansion step (updates the node arrays [B, cap] in place).
    frontier [B, F] node ids; topk_tok / topk_prob_ [B, F, k].  Returns
    (next frontier [B, k_next] node ids, near [B] bool)."""
    fr = _i32(frontier)
    B, F = fr.shape
    tt = _i32(topk_tok).reshape(B, F, -1)
    k = tt.shape[2]
    tp = np.ascontiguousarray(topk_prob_, dtype=np.float64).reshape(B, F, k)
    for arr, dt in ((node_tok, np.int32), (node_val, np.float64), (node_par, np.int32)):
        if not (isinstance(arr, np.ndarray) and arr.dtype == dt and arr.flags.c_contiguous):
            raise TypeError("node arrays must be contiguous numpy arrays (int32, float64, int32)")
    cap = node_tok.shape[1]
    out = np.zeros((B, k_next), dtype=np.int32)
    near = np.zeros(B, dtype=np.uint8)
    st = _load().oracle_eagle2_expand(_ptr(fr), B, F, k, _ptr(tt), _ptr(tp), _ptr(node_tok), _ptr(node_val),
                                      _ptr(node_par), cap, int(offset), int(k_next), _ptr(out), _ptr(near))
    if st != OK:
        raise ValueError("oracle_eagle2_expand: invalid arguments")
    return out, near.astype(bool)


def eagle2_rerank(node_val, node_par, node_tok, m: int):
    """Keep the root and the m best nodes of each of B trees [B, M].  Returns
    (parent [B, m+1] as list positions, tokens [B, m+1], node ids [B, m+1],
    near [B] bool)."""
    val = np.ascontiguousarray(node_val, dtype=np.float64)
    par = _i32(node_par)
    tok = _i32(node_tok)
    B, M = val.shape
    op = np.zeros((B, m + 1), dtype=np.int32)
    ot = np.zeros((B, m + 1), dtype=np.int32)
    oi = np.zeros((B, m + 1), dtype=np.int32)
    near = np.zeros(B, dtype=np.uint8)
    st = _load().oracle_eagle2_rerank(_ptr(val), _ptr(par), _ptr(tok), B, M, int(m), _ptr(op), _ptr(ot),
                                      _ptr(oi), _ptr(near))
    if st == ERR_PARENT:
        raise ValueError("oracle_eagle2_rerank: malformed tree or a kept node's parent was dropped")
    if st != OK:
        raise ValueError("oracle_eagle2_rerank: invalid arguments")
    return op, ot, oi, near.astype(bool)


def verify_points(zt, x, counts, T: float, seed: int, *, b_ids=None, nthreads=1):
    """Verification of point-mass drafts (a deterministic drafter such as the
    n-gram drafter): zt [nb, K+1, V], x [nb, K], counts [nb] or None (all K).
    Returns a dict with tokens [nb, K+1], n [nb], near [nb] bool, status."""
    zt_a, dt = _logits(zt)
    nb, K1, V = zt_a.shape
    K = K1 - 1
    xs = _i32(x).reshape(nb, K)
    cn = None if counts is None else _i32(counts).reshape(nb)
    bi = None if b_ids is None else _i32(b_ids).reshape(nb)
    tokens = np.zeros((nb, K + 1), dtype=np.int32)
    n = np.zeros(nb, dtype=np.int32)
    near = np.zeros(nb, dtype=np.int32)
    st = _load().oracle_verify_points(_ptr(zt_a), _ptr(xs), _ptr(cn), nb, K, V, dt, float(T),
                                      int(seed) & ((1 << 64) - 1), _ptr(bi), _ptr(tokens), _ptr(n), _ptr(near),
                                      int(nthreads))
    if st == ERR_ARG:
        raise ValueError("oracle_verify_points: invalid arguments")
    return dict(tokens=tokens, n=n, near=near.astype(bool), status=st)
