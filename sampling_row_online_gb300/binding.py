"""Thin ctypes binding of libspec_verify.so (argument marshalling only).

Every step of the verification runs in the library's CUDA kernels; this module
checks tensor shapes, dtypes and devices, passes raw device pointers and the
current CUDA stream, and raises ``SpecError`` on a non-zero status.  There is
no fallback: if the library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SPEC_OK = 0
SPEC_F32, SPEC_BF16 = 0, 1
STATUS_NAMES = {
    0: "SPEC_OK", 1: "SPEC_ERR_ARG", 2: "SPEC_ERR_DTYPE", 3: "SPEC_ERR_ALIGN",
    4: "SPEC_ERR_TOKEN_RANGE", 5: "SPEC_ERR_CUDA", 6: "SPEC_ERR_TIMEOUT",
    7: "SPEC_ERR_PARENT", 8: "SPEC_ERR_UNSUPPORTED",
}

_lib = None


class SpecError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(abs(status), f"status {status}")
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class StatsStruct(ctypes.Structure):
    _fields_ = [(n, ctypes.c_ulonglong) for n in
                ("sequences", "accepted", "bonus", "resampled", "residual_fallbacks", "errors",
                 "near_boundary")]

STATS_COUNTERS = len(StatsStruct._fields_)


def library():
    """Loads libspec_verify.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        path = _build.build()
    lib = ctypes.CDLL(path)
    vp, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    lib.spec_verify.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp]
    lib.spec_verify_ex.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_host.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp]
    lib.spec_arm_rows_event.argtypes = [vp]
    lib.spec_arm_timer.argtypes = [vp]
    lib.spec_verify_tree_greedy.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.spec_verify_tree.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, u64, i32, vp, vp, vp]
    lib.spec_verify_trees_greedy.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.spec_verify_trees.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, u64, i32, vp, vp, vp]
    lib.spec_tree_max_depth.argtypes = [vp, i32]
    lib.spec_tree_mask.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.spec_ngram_propose.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.spec_topk.argtypes = [vp, i32, i32, i32, f32, i32, vp, vp, vp]
    lib.spec_selftest_wait.argtypes = [vp]
    lib.spec_debug_fail_launch.argtypes = [i32]
    lib.spec_verify_points.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp]
    lib.spec_eagle2_expand.argtypes = [vp, vp, i32, i32, i32, i32, f32, i32, vp, vp, vp, i32, i32, i32, vp, vp]
    lib.spec_eagle2_rerank.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp]
    lib.spec_get_status.argtypes = [vp]
    lib.spec_error_string.argtypes = [i32]
    lib.spec_error_string.restype = ctypes.c_char_p
    lib.spec_last_error_message.argtypes = []
    lib.spec_last_error_message.restype = ctypes.c_char_p
    lib.spec_verify_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp]
    lib.spec_noalloc_get_status.argtypes = [vp]
    lib.spec_debug_noalloc_status.argtypes = [i32]
    lib.spec_shutdown.argtypes = []
    lib.spec_shutdown.restype = None
    for name in ("spec_verify", "spec_verify_ex", "spec_verify_host", "spec_verify_tree_greedy",
                 "spec_tree_max_depth", "spec_tree_mask", "spec_ngram_propose", "spec_topk",
                 "spec_eagle2_expand", "spec_eagle2_rerank", "spec_get_status", "spec_verify_noalloc",
                 "spec_noalloc_get_status", "spec_debug_noalloc_status"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != SPEC_OK:
        detail = library().spec_last_error_message().decode(errors="replace")
        raise SpecError(status, where, detail)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _chain_shapes(target_logits, draft_logits, draft_tokens):
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if draft_tokens is not None and tuple(draft_tokens.shape) != (B, K):
        raise ValueError(f"draft_tokens must be [B, K] = [{B}, {K}]")
    if draft_logits is not None and K > 0:
        if tuple(draft_logits.shape) != (B, K, V) or draft_logits.dtype != target_logits.dtype:
            raise ValueError(f"draft_logits must be [B, K, V] = [{B}, {K}, {V}] of the target dtype")
    return B, K, V


def spec_verify(target_logits, draft_logits, draft_tokens, temperature, seed, *,
                out_tokens=None, out_n_accepted=None, stream=None):
    """Chain verification; returns (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    return spec_verify_ex(target_logits, draft_logits, draft_tokens, temperature, seed,
                          out_tokens=out_tokens, out_n_accepted=out_n_accepted,
                          stream=stream)[:2]


def spec_verify_ex(target_logits, draft_logits, draft_tokens, temperature, seed, *,
                   out_tokens=None, out_n_accepted=None, want_row_stats=False, stats=None,
                   stream=None):
    """Chain verification with optional per-row (max, sumexp) [B, 2K+1] outputs and a
    device ``stats`` tensor (STATS_COUNTERS int64 counters, accumulated).  Returns
    (out_tokens, n_accepted, row_max or None, row_sumexp or None)."""
    lib = library()
    _dev(target_logits, "target_logits")
    B, K, V = _chain_shapes(target_logits, draft_logits, draft_tokens)
    _dev(draft_logits, "draft_logits")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(out_tokens, "out_tokens", torch.int32)
    _dev(out_n_accepted, "out_n_accepted", torch.int32)
    row_max = row_sumexp = None
    if want_row_stats:
        row_max = torch.empty((B, 2 * K + 1), dtype=torch.float32, device=dev)
        row_sumexp = torch.empty((B, 2 * K + 1), dtype=torch.float32, device=dev)
    if stats is not None:
        _dev(stats, "stats", torch.int64)
        if stats.numel() != STATS_COUNTERS:
            raise ValueError(f"stats must hold {STATS_COUNTERS} int64 counters")
    with torch.cuda.device(dev):
        st = lib.spec_verify_ex(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens),
                                B, K, V, _dtype_code(target_logits), float(temperature),
                                int(seed) & (2 ** 64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
                                _ptr(row_max), _ptr(row_sumexp), _ptr(stats), _stream(stream))
    _check(st, "spec_verify")
    return out_tokens, out_n_accepted, row_max, row_sumexp


def spec_verify_host(target_logits, draft_logits, draft_tokens, temperature, seed, *,
                     out_tokens=None, out_n_accepted=None, device=None, stream=None):
    """End-to-end chain verification on HOST (CPU) tensors: the library copies the
    inputs to the GPU, verifies, copies the outputs back and waits.  Pinned host
    tensors give the fastest copies.  Returns (out_tokens, n_accepted) on the host."""
    lib = library()
    for t, name in ((target_logits, "target_logits"), (draft_logits, "draft_logits"),
                    (draft_tokens, "draft_tokens")):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    B, K, V = _chain_shapes(target_logits, draft_logits, draft_tokens)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, pin_memory=True)
    if out_n_accepted is None:
        out_n_accepted = torch.empty((B,), dtype=torch.int32, pin_memory=True)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        st = lib.spec_verify_host(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens),
                                  B, K, V, _dtype_code(target_logits), float(temperature),
                                  int(seed) & (2 ** 64 - 1), _ptr(out_tokens),
                                  _ptr(out_n_accepted), _stream(stream))
    _check(st, "spec_verify_host")
    return out_tokens, out_n_accepted


def spec_tree_max_depth(parent) -> int:
    """Largest node depth of parent[] (host data)."""
    p = torch.as_tensor(parent, dtype=torch.int32).contiguous().cpu()
    d = library().spec_tree_max_depth(_ptr(p), p.numel())
    if d < 0:
        _check(-d, "spec_tree_max_depth")
    return d


def _tree_parents(parent, B, N, max_depth):
    """(one tree per sequence?, max_depth) for a parent tensor [N] (one tree)
    or [B, N]; a missing max_depth is the deepest node over the trees (read
    on the host)."""
    if parent.dim() == 2:
        if tuple(parent.shape) != (B, N):
            raise ValueError("parent must be [N] or [B, N]")
        if max_depth is None:
            max_depth = max((spec_tree_max_depth(row) for row in parent.cpu()), default=0)
        return True, max_depth
    if parent.numel() != N:
        raise ValueError("parent must be [N] or [B, N]")
    return False, spec_tree_max_depth(parent.cpu()) if max_depth is None else max_depth


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, temperature, seed, *,
                        out_tokens=None, out_n_accepted=None, stream=None):
    """Chain verification on the library's fixed scratch (no device allocation
    in the call; calls that overlap on the GPU must be serialised).  Returns
    (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    lib = library()
    _dev(target_logits, "target_logits")
    B, K, V = _chain_shapes(target_logits, draft_logits, draft_tokens)
    _dev(draft_logits, "draft_logits")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev(out_tokens, "out_tokens", torch.int32)
    _dev(out_n_accepted, "out_n_accepted", torch.int32)
    with torch.cuda.device(dev):
        st = lib.spec_verify_noalloc(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, K, V,
                                     _dtype_code(target_logits), float(temperature), int(seed) & (2 ** 64 - 1),
                                     _ptr(out_tokens), _ptr(out_n_accepted), _stream(stream))
    _check(st, "spec_verify_noalloc")
    return out_tokens, out_n_accepted


def spec_verify_tree_greedy(target_logits, parent, node_tokens, *, max_depth=None,
                            out_path=None, out_len=None, stream=None):
    """Greedy tree verification; parent [N] (one tree) or [B, N] (one tree per
    sequence).  Returns (out_path [B, D+1] int32, out_len [B] int32)."""
    lib = library()
    _dev(target_logits, "target_logits")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = target_logits.shape
    _dev(parent, "parent", torch.int32)
    _dev(node_tokens, "node_tokens", torch.int32)
    if tuple(node_tokens.shape) != (B, N):
        raise ValueError("node_tokens must be [B, N]")
    per_seq, max_depth = _tree_parents(parent, B, N, max_depth)
    dev = target_logits.device
    if out_path is None:
        out_path = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    fn = lib.spec_verify_trees_greedy if per_seq else lib.spec_verify_tree_greedy
    with torch.cuda.device(dev):
        st = fn(_ptr(target_logits), _ptr(parent), _ptr(node_tokens),
                                         B, N, V, _dtype_code(target_logits), int(max_depth),
                                         _ptr(out_path), _ptr(out_len), _stream(stream))
    _check(st, "spec_verify_tree_greedy")
    return out_path, out_len


def spec_verify_tree(target_logits, draft_logits, parent, node_tokens, temperature, seed, *,
                     max_depth=None, out_path=None, out_len=None, stream=None):
    """Stochastic tree verification (T > 0; T == 0 is greedy matching); parent
    [N] (one tree) or [B, N] (one tree per sequence).  Returns (out_path
    [B, D+1] int32, out_len [B] int32)."""
    lib = library()
    _dev(target_logits, "target_logits")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = target_logits.shape
    if draft_logits is not None:
        _dev(draft_logits, "draft_logits", target_logits.dtype)
        if tuple(draft_logits.shape) != (B, N, V):
            raise ValueError("draft_logits must be [B, N, V]")
    _dev(parent, "parent", torch.int32)
    _dev(node_tokens, "node_tokens", torch.int32)
    if tuple(node_tokens.shape) != (B, N):
        raise ValueError("node_tokens must be [B, N]")
    per_seq, max_depth = _tree_parents(parent, B, N, max_depth)
    dev = target_logits.device
    if out_path is None:
        out_path = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    fn = lib.spec_verify_trees if per_seq else lib.spec_verify_tree
    with torch.cuda.device(dev):
        st = fn(_ptr(target_logits), _ptr(draft_logits), _ptr(parent),
                                  _ptr(node_tokens), B, N, V, _dtype_code(target_logits),
                                  ctypes.c_float(temperature), ctypes.c_uint64(int(seed) & ((1 << 64) - 1)),
                                  int(max_depth), _ptr(out_path), _ptr(out_len), _stream(stream))
    _check(st, "spec_verify_tree")
    return out_path, out_len


def spec_verify_trees_greedy(target_logits, parent, node_tokens, *, max_depth=None, out_path=None,
                             out_len=None, stream=None):
    """Greedy verification of one tree per sequence: parent [B, N] int32.
    Returns (out_path [B, D+1] int32, out_len [B] int32)."""
    if parent.dim() != 2:
        raise ValueError("parent must be [B, N] (one tree per sequence)")
    return spec_verify_tree_greedy(target_logits, parent, node_tokens, max_depth=max_depth, out_path=out_path,
                                   out_len=out_len, stream=stream)


def spec_verify_trees(target_logits, draft_logits, parent, node_tokens, temperature, seed, *, max_depth=None,
                      out_path=None, out_len=None, stream=None):
    """Stochastic verification of one tree per sequence: parent [B, N] int32.
    Returns (out_path [B, D+1] int32, out_len [B] int32)."""
    if parent.dim() != 2:
        raise ValueError("parent must be [B, N] (one tree per sequence)")
    return spec_verify_tree(target_logits, draft_logits, parent, node_tokens, temperature, seed,
                            max_depth=max_depth, out_path=out_path, out_len=out_len, stream=stream)


def spec_tree_mask(parent, *, stream=None):
    """Tree-attention masks and depth position IDs of B trees.

    parent: [B, N] int32 CUDA tensor.  Returns (mask [B, N, ceil(N/32)] int32 bit
    words, depth [B, N] int32)."""
    lib = library()
    _dev(parent, "parent", torch.int32)
    if parent.dim() == 1:
        parent = parent.unsqueeze(0)
    B, N = parent.shape
    W = (N + 31) // 32
    mask = torch.empty((B, N, W), dtype=torch.int32, device=parent.device)
    depth = torch.empty((B, N), dtype=torch.int32, device=parent.device)
    with torch.cuda.device(parent.device):
        st = lib.spec_tree_mask(_ptr(parent), B, N, _ptr(mask), _ptr(depth), _stream(stream))
    _check(st, "spec_tree_mask")
    return mask, depth


def spec_verify_points(target_logits, draft_tokens, temperature, seed, *, draft_counts=None, out_tokens=None,
                       out_n=None, stream=None):
    """Chain verification of point-mass drafts (a deterministic drafter such as
    spec_ngram_propose).  target_logits [B, K+1, V]; draft_tokens [B, K] int32;
    draft_counts [B] int32 or None (all K).  Returns (out_tokens [B, K+1],
    n_accepted [B])."""
    lib = library()
    _dev(target_logits, "target_logits")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if tuple(draft_tokens.shape) != (B, K):
        raise ValueError("draft_tokens must be [B, K]")
    if draft_counts is not None:
        _dev(draft_counts, "draft_counts", torch.int32)
        if tuple(draft_counts.shape) != (B,):
            raise ValueError("draft_counts must be [B]")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = lib.spec_verify_points(_ptr(target_logits), _ptr(draft_tokens), _ptr(draft_counts), B, K, V,
                                    _dtype_code(target_logits), ctypes.c_float(temperature),
                                    ctypes.c_uint64(int(seed) & ((1 << 64) - 1)), _ptr(out_tokens), _ptr(out_n),
                                    _stream(stream))
    _check(st, "spec_verify_points")
    return out_tokens, out_n


def spec_ngram_propose(tokens, lengths, n_min, n_max, K, *, min_hits=1, out_draft=None, out_count=None,
                       stream=None):
    """n-gram (prompt-lookup) drafts of B contexts.

    tokens: [B, L] int32 CUDA tensor (row b's context in its first lengths[b]
    entries); lengths: [B] int32.  Returns (draft [B, K] int32, -1 after the
    proposal; count [B] int32, 0 = no match)."""
    lib = library()
    _dev(tokens, "tokens", torch.int32)
    _dev(lengths, "lengths", torch.int32)
    if tokens.dim() != 2:
        raise ValueError("tokens must be [B, L]")
    B, L = tokens.shape
    if lengths.shape != (B,):
        raise ValueError("lengths must be [B]")
    if out_draft is None:
        out_draft = torch.empty((B, K), dtype=torch.int32, device=tokens.device)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=tokens.device)
    _dev(out_draft, "out_draft", torch.int32)
    _dev(out_count, "out_count", torch.int32)
    if out_draft.shape != (B, K) or out_count.shape != (B,):
        raise ValueError("out_draft must be [B, K] and out_count [B]")
    with torch.cuda.device(tokens.device):
        st = lib.spec_ngram_propose(_ptr(tokens), _ptr(lengths), B, L, int(n_min), int(n_max), int(min_hits),
                                    int(K), _ptr(out_draft), _ptr(out_count), _stream(stream))
    _check(st, "spec_ngram_propose")
    return out_draft, out_count


def spec_topk(logits, k, temperature=1.0, *, out_tokens=None, out_prob=None, stream=None):
    """Top-k tokens of each row of logits [..., V] (ties to the lower index)
    and their probabilities under softmax(z / T).  Returns (tokens [R, k]
    int32, prob [R, k] float32) with R the number of rows."""
    lib = library()
    _dev(logits, "logits")
    V = logits.shape[-1]
    R = logits.numel() // V if V else 0
    if out_tokens is None:
        out_tokens = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    if out_prob is None:
        out_prob = torch.empty((R, k), dtype=torch.float32, device=logits.device)
    with torch.cuda.device(logits.device):
        st = lib.spec_topk(_ptr(logits), R, V, _dtype_code(logits), float(temperature), int(k), _ptr(out_tokens),
                           _ptr(out_prob), _stream(stream))
    _check(st, "spec_topk")
    return out_tokens, out_prob


def spec_eagle2_expand(draft_logits, frontier, node_tokens, node_values, node_parents, k, offset, k_next,
                       temperature=1.0, *, out_frontier=None, stream=None):
    """One EAGLE-2 expansion step.  draft_logits [B, F, V]; frontier [B, F]
    int32 node ids; node arrays [B, cap] (int32 tokens, float32 values, int32
    parents; node 0 the root), updated in place at nodes offset ..
    offset + F*k - 1.  Returns the next frontier [B, k_next] int32."""
    lib = library()
    _dev(draft_logits, "draft_logits")
    _dev(frontier, "frontier", torch.int32)
    _dev(node_tokens, "node_tokens", torch.int32)
    _dev(node_values, "node_values", torch.float32)
    _dev(node_parents, "node_parents", torch.int32)
    if draft_logits.dim() != 3:
        raise ValueError("draft_logits must be [B, F, V]")
    B, F, V = draft_logits.shape
    cap = node_tokens.shape[1]
    if frontier.shape != (B, F) or node_values.shape != (B, cap) or node_parents.shape != (B, cap):
        raise ValueError("frontier must be [B, F] and the node arrays [B, cap]")
    if out_frontier is None:
        out_frontier = torch.empty((B, k_next), dtype=torch.int32, device=draft_logits.device)
    with torch.cuda.device(draft_logits.device):
        st = lib.spec_eagle2_expand(_ptr(draft_logits), _ptr(frontier), B, F, V, _dtype_code(draft_logits),
                                    float(temperature), int(k), _ptr(node_tokens), _ptr(node_values),
                                    _ptr(node_parents), cap, int(offset), int(k_next), _ptr(out_frontier),
                                    _stream(stream))
    _check(st, "spec_eagle2_expand")
    return out_frontier


def spec_eagle2_rerank(node_values, node_parents, node_tokens, m, *, stream=None):
    """EAGLE-2 rerank of B trees [B, M]: the root and the m best nodes listed
    by depth.  Returns (parent [B, m+1] list positions, tokens [B, m+1],
    node ids [B, m+1]), all int32."""
    lib = library()
    _dev(node_values, "node_values", torch.float32)
    _dev(node_parents, "node_parents", torch.int32)
    _dev(node_tokens, "node_tokens", torch.int32)
    B, M = node_values.shape
    dev = node_values.device
    out = [torch.empty((B, m + 1), dtype=torch.int32, device=dev) for _ in range(3)]
    with torch.cuda.device(dev):
        st = lib.spec_eagle2_rerank(_ptr(node_values), _ptr(node_parents), _ptr(node_tokens), B, M, int(m),
                                    _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), _stream(stream))
    _check(st, "spec_eagle2_rerank")
    return tuple(out)


def spec_selftest_wait(stream=None) -> int:
    """Launches the bounded-wait self-test on the stream and returns the status
    the next spec_get_status reports (SPEC_ERR_TIMEOUT when the wait ended by
    its limit, after about a second)."""
    _check(library().spec_selftest_wait(_stream(stream)), "spec_selftest_wait")
    return spec_get_status(stream)


def spec_get_status(stream=None) -> int:
    """Waits for the stream; returns (and clears) the device-side status code."""
    return int(library().spec_get_status(_stream(stream)))


def spec_noalloc_get_status(stream=None) -> int:
    """Waits for the stream; returns (and clears) the status code recorded in
    the fixed array of spec_verify_noalloc."""
    return int(library().spec_noalloc_get_status(_stream(stream)))


def spec_debug_noalloc_status(bits):
    """Test hook: ORs device status bits (1 token out of range, 4 a wait ran
    out) into the status word of spec_verify_noalloc's fixed array."""
    _check(library().spec_debug_noalloc_status(int(bits)), "spec_debug_noalloc_status")


def raise_on_device_error(stream=None):
    st = spec_get_status(stream)
    _check(st, "device")


def spec_arm_rows_event(event):
    """Measurement hook: the next verification call made from this thread
    records `event` (a torch.cuda.Event that has been recorded once, so that
    it exists) between its streaming and decision kernels."""
    library().spec_arm_rows_event(ctypes.c_void_p(event.cuda_event))


def spec_arm_timer(stamps):
    """Measurement hook: the next verification call made from this thread
    records global-timer stamps into `stamps` (a CUDA int64 tensor of 3 words
    set to (-1, 0, 0), read as unsigned): first streaming-CTA start, last
    streaming-CTA end, last output."""
    _dev(stamps, "stamps", torch.int64)
    if stamps.numel() < 3:
        raise ValueError("stamps must hold 3 int64 words")
    library().spec_arm_timer(_ptr(stamps))


def spec_debug_fail_launch(n):
    """Fault injection: the n-th next kernel launch of the library fails with a
    launch error (n = 0 switches it off)."""
    _check(library().spec_debug_fail_launch(int(n)), "spec_debug_fail_launch")


def spec_error_string(status):
    return library().spec_error_string(int(status)).decode()


def spec_last_error_message():
    return library().spec_last_error_message().decode(errors="replace")


def spec_shutdown():
    """Frees every workspace the library holds (no call may be in flight)."""
    library().spec_shutdown()
