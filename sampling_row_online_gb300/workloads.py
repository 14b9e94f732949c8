"""Seeded synthetic inputs for the verification step.

This module only *generates inputs*: logits with the distributions of the
workloads below, draft tokens drawn the way a drafter would draw them, and the
static draft tree.  It holds none of the verification arithmetic (no
normalisers, no acceptance test, no residual, no inverse CDF): the same tensors
are fed to the CUDA library and to the fp64 oracle, and only those two compute
the method.

Draft tokens are drawn from softmax(z_d / T) with the Gumbel-max trick
(argmax of z_d / T + Gumbel noise), using torch's seeded generator on the
device the tensors live on.  Node tokens of the tree workload equal the
target's top token of the parent row with probability ``p_correct`` and are
uniform otherwise.

Workloads (sizes are those of the benchmark and the parity tests):

====  =========  ====  ===  =======  =====  ====  =======================================
name  kind       B     K/N  V        dtype  T     logits
====  =========  ====  ===  =======  =====  ====  =======================================
c0    chain      1     4    32000    f32    1.0   z_t ~ N(0, 3^2); z_d = z_t + N(0, 1)
c1    chain      64    5    128256   bf16   0.7   z_t ~ N(0, 3^2); z_d = z_t + N(0, 0.5^2)
c2    chain      256   8    151936   bf16   1.0   z_t ~ N(0, 4^2); z_d = z_t + N(0, 2^2)
c3    tree       32    63   128256   bf16   0     z_t ~ N(0, 3^2); static tree 4/3/2/2/1
c4    chain      512   4    256000   f32    1.0   z_t = 1.5 * (-1.1 ln rank) + N(0, 1);
                                                  z_d = z_t + N(0, 1)
====  =========  ====  ===  =======  =====  ====  =======================================

n-gram drafting contexts (``NGRAM_WORKLOADS``, ``make_contexts``): B rows of
up to L tokens, lengths uniform in [L/2, L].  A row is a sequence of segments
(geometric lengths, mean ``mean_seg``); a segment either holds fresh tokens
(log-uniform ranks over V, i.e. Zipf with exponent 1) or, with probability
``copy_frac``, repeats the span that starts d tokens earlier (d uniform over
the positions before the segment), as when code or a cited source is edited.

====  ===  =====  ===========  ========  ==
name  B    L      n_min..n_max  min_hits  K
====  ===  =====  ===========  ========  ==
ng1   64   32768  1..4          1         5
ng2   64   32768  8..8          2         5
====  ===  =====  ===========  ========  ==

EAGLE-2 tree budget (``EAGLE2_WORKLOADS``): a stand-in draft model whose
logits at a node are sigma * N(0, 1) over V from a generator seeded by the
node's token path (``node_key``), so that any two callers that reach the same
node see the same row; ``eagle2_step_rows`` gives the bench its per-step row
tensors directly.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "chain" or "tree"
    B: int
    K: int               # drafts per sequence (chain); nodes N (tree)
    V: int
    dtype: str           # "f32" or "bf16"
    T: float
    sigma_t: float = 3.0
    sigma_d: float = 1.0
    zipf: bool = False
    p_correct: float = 0.6
    branching: tuple = field(default=(4, 3, 2, 2, 1))
    data_seed: int = 1000
    verify_seed: int = 0
    draft_seed: int | None = None

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def N(self) -> int:
        return self.K

    @property
    def rows(self) -> int:
        """Logit rows one call reads: (2K+1) per sequence for a stochastic chain,
        K+1 for a greedy chain, N for a tree, N plus one draft row per node with
        children for a stochastic tree."""
        if self.kind == "tree":
            return self.B * self.K
        if self.kind == "tree_sample":
            parent = tree_parents(self.branching, self.K)
            return self.B * (self.K + len(set(parent[1:])))
        if self.T == 0:
            return self.B * (self.K + 1)
        return self.B * (2 * self.K + 1)

    @property
    def algorithmic_bytes(self) -> int:
        """Every logit the data-parallel step must read once."""
        return self.rows * self.V * self.elem_bytes

    @property
    def positions(self) -> int:
        """Verified draft positions per call: B*K (chain), B*(N-1) (tree)."""
        return self.B * (self.K - 1) if self.kind in ("tree", "tree_sample") else self.B * self.K

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "c0": Workload("c0", "chain", B=1, K=4, V=32000, dtype="f32", T=1.0,
                   sigma_t=3.0, sigma_d=1.0, data_seed=1000, verify_seed=0, draft_seed=0),
    "c1": Workload("c1", "chain", B=64, K=5, V=128256, dtype="bf16", T=0.7,
                   sigma_t=3.0, sigma_d=0.5, data_seed=1001, verify_seed=1),
    "c2": Workload("c2", "chain", B=256, K=8, V=151936, dtype="bf16", T=1.0,
                   sigma_t=4.0, sigma_d=2.0, data_seed=1002, verify_seed=2),
    "c3": Workload("c3", "tree", B=32, K=63, V=128256, dtype="bf16", T=0.0,
                   sigma_t=3.0, data_seed=1003, verify_seed=3),
    "c4": Workload("c4", "chain", B=512, K=4, V=256000, dtype="f32", T=1.0,
                   sigma_t=1.0, sigma_d=1.0, zipf=True, data_seed=1004, verify_seed=4),
    # not one of the headline configurations: the tree of c3 verified
    # stochastically, candidates drawn from the draft at their parent
    "c3s": Workload("c3s", "tree_sample", B=32, K=63, V=128256, dtype="bf16", T=1.0,
                    sigma_t=3.0, sigma_d=1.0, data_seed=1005, verify_seed=5),
}


def describe(w: Workload) -> str:
    if w.kind == "tree":
        return (f"tree B={w.B} N={w.K} V={w.V} {w.dtype} T=0 "
                f"branching={'/'.join(map(str, w.branching))}")
    if w.kind == "tree_sample":
        return (f"stochastic tree B={w.B} N={w.K} V={w.V} {w.dtype} T={w.T} "
                f"branching={'/'.join(map(str, w.branching))}")
    return f"chain B={w.B} K={w.K} V={w.V} {w.dtype} T={w.T}"


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def tree_parents(branching=(4, 3, 2, 2, 1), N=63):
    """Static draft tree in breadth-first order: every node of level l gets
    branching[l] children, levels are filled left to right, and the tree is cut
    at N nodes.  Returns parent[] with parent[0] = -1 and parent[c] < c."""
    parent = [-1]
    level = [0]
    for b in branching:
        nxt = []
        for p in level:
            for _ in range(b):
                if len(parent) == N:
                    break
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
        if len(parent) == N:
            break
    return parent


def gumbel_argmax_draws(logits_scaled: torch.Tensor, g: torch.Generator, chunk_rows=256):
    """Index draws from softmax(logits_scaled) per row, by the Gumbel-max trick.

    logits_scaled: [R, V] float32.  Each row's draw is argmax(x + G), G iid
    standard Gumbel from the seeded generator."""
    R, V = logits_scaled.shape
    out = torch.empty(R, dtype=torch.int32, device=logits_scaled.device)
    for r0 in range(0, R, chunk_rows):
        x = logits_scaled[r0:r0 + chunk_rows]
        u = torch.rand(x.shape, generator=g, device=x.device, dtype=torch.float64)
        u = u.clamp_(min=1e-300, max=1.0 - 1e-16)
        gum = -torch.log(-torch.log(u))
        out[r0:r0 + chunk_rows] = torch.argmax(x.double() + gum, dim=-1).to(torch.int32)
    return out


def make_chain(w: Workload, device="cpu", *, with_draft_logits=True):
    """(target_logits [B,K+1,V], draft_logits [B,K,V] or None, draft_tokens [B,K] int32)."""
    assert w.kind == "chain"
    g = _gen(device, w.data_seed)
    B, K, V = w.B, w.K, w.V
    if w.zipf:
        perm = torch.randperm(V, generator=g, device=device)
        bias = 1.5 * (-1.1 * torch.log((perm + 1).to(torch.float32)))
        zt32 = torch.randn((B, K + 1, V), generator=g, device=device) * w.sigma_t + bias
    else:
        zt32 = torch.randn((B, K + 1, V), generator=g, device=device) * w.sigma_t
    zt = zt32.to(w.torch_dtype)
    zd = None
    if K > 0 and (with_draft_logits or w.T > 0):
        zd32 = zt32[:, :K] + torch.randn((B, K, V), generator=g, device=device) * w.sigma_d
        del zt32
        zd = zd32.to(w.torch_dtype)
        del zd32
    else:
        del zt32
    # draft tokens: what the drafter sampled from q = softmax(z_d / T)
    gd = _gen(device, w.draft_seed if w.draft_seed is not None else w.data_seed + 7919)
    if K == 0:
        x = torch.zeros((B, 0), dtype=torch.int32, device=device)
    elif zd is not None and w.T > 0:
        x = gumbel_argmax_draws(zd.reshape(B * K, V).float() / w.T, gd).reshape(B, K)
    elif zd is not None:
        x = torch.argmax(zd.reshape(B * K, V).float(), dim=-1).to(torch.int32).reshape(B, K)
    else:
        x = torch.randint(0, V, (B, K), generator=gd, device=device, dtype=torch.int32)
    return zt, zd, x.contiguous()


def make_tree(w: Workload, device="cpu"):
    """(target_logits [B,N,V], parent [N] int32, node_tokens [B,N] int32)."""
    assert w.kind == "tree"
    g = _gen(device, w.data_seed)
    B, N, V = w.B, w.K, w.V
    zt = (torch.randn((B, N, V), generator=g, device=device) * w.sigma_t).to(w.torch_dtype)
    parent = torch.tensor(tree_parents(w.branching, N), dtype=torch.int32, device=device)
    top = torch.argmax(zt.float(), dim=-1).to(torch.int32)              # [B, N]
    top_of_parent = top[:, parent.clamp(min=0).long()]                  # [B, N]
    coin = torch.rand((B, N), generator=g, device=device) < w.p_correct
    rnd = torch.randint(0, V, (B, N), generator=g, device=device, dtype=torch.int32)
    tok = torch.where(coin, top_of_parent, rnd)
    tok[:, 0] = 0
    return zt, parent, tok.contiguous()


def make_tree_sample(w: Workload, device="cpu"):
    """(target_logits [B,N,V], draft_logits [B,N,V], parent [N] int32,
    node_tokens [B,N] int32) of a stochastic tree: z_d = z_t + N(0, sigma_d^2),
    and the candidates of every node drawn independently from
    softmax(z_d[parent] / T) (what a drafter sampling the tree would do)."""
    assert w.kind == "tree_sample"
    g = _gen(device, w.data_seed)
    B, N, V = w.B, w.K, w.V
    zt32 = torch.randn((B, N, V), generator=g, device=device) * w.sigma_t
    zd32 = zt32 + torch.randn((B, N, V), generator=g, device=device) * w.sigma_d
    zt = zt32.to(w.torch_dtype)
    del zt32
    zd = zd32.to(w.torch_dtype)
    del zd32
    parent = torch.tensor(tree_parents(w.branching, N), dtype=torch.int32, device=device)
    tok = torch.zeros((B, N), dtype=torch.int32, device=device)
    if N > 1:
        gd = _gen(device, w.data_seed + 7919)
        rows = zd[:, parent[1:].long()].reshape(B * (N - 1), V).float() / w.T
        tok[:, 1:] = gumbel_argmax_draws(rows, gd).reshape(B, N - 1)
    return zt, zd, parent, tok.contiguous()


def input_copies_for_cold_l2(bytes_per_copy: int, l2_bytes: int = 129 * 2**20) -> int:
    """Number of input copies to rotate so that consecutive calls never find
    their inputs in L2: the copies together exceed twice the L2 size."""
    return max(2, math.ceil(2 * l2_bytes / max(1, bytes_per_copy)) + 1)


@dataclass(frozen=True)
class NgramWorkload:
    name: str
    B: int
    L: int               # row capacity: the longest context
    n_min: int
    n_max: int
    min_hits: int
    K: int
    V: int = 128256
    copy_frac: float = 0.5
    mean_seg: int = 24
    data_seed: int = 2000

    @property
    def context_bytes(self) -> int:
        return self.B * self.L * 4


NGRAM_WORKLOADS = {
    # vLLM's n-gram settings on the pages: K = 5 speculative tokens, n-gram window up to 4
    "ng1": NgramWorkload("ng1", B=64, L=32768, n_min=1, n_max=4, min_hits=1, K=5, data_seed=2001),
    # llama.cpp's setting for text on the pages: n = 8, min-hits 2
    "ng2": NgramWorkload("ng2", B=64, L=32768, n_min=8, n_max=8, min_hits=2, K=5, data_seed=2002),
}


def make_contexts(w: NgramWorkload, device="cpu", *, B=None, L=None, seed=None):
    """(tokens [B, L] int32, lengths [B] int32) on ``device``; entries past a
    row's length are filled too (with the same process), so that nothing
    depends on them being ignored."""
    B = w.B if B is None else B
    L = w.L if L is None else L
    g = _gen(device, w.data_seed if seed is None else seed)
    if B == 0 or L == 0:
        return (torch.zeros((B, L), dtype=torch.int32, device=device),
                torch.zeros((B,), dtype=torch.int32, device=device))
    u = torch.rand((B, L), generator=g, device=device, dtype=torch.float64)
    fresh = torch.floor(torch.exp(u * math.log(w.V))).clamp_(1, w.V).long() - 1
    pos = torch.arange(L, device=device).expand(B, L)
    starts = torch.rand((B, L), generator=g, device=device) < 1.0 / w.mean_seg
    starts[:, 0] = True
    seg_start = torch.cummax(torch.where(starts, pos, torch.zeros_like(pos)), dim=1).values
    u_copy = torch.rand((B, L), generator=g, device=device).gather(1, seg_start)
    u_off = torch.rand((B, L), generator=g, device=device, dtype=torch.float64).gather(1, seg_start)
    copy = (u_copy < w.copy_frac) & (seg_start > 0)
    d = 1 + torch.floor(u_off * seg_start).long()           # 1 <= d <= seg_start
    src = torch.where(copy, pos - d, pos)                  # src[i] < i on copied positions
    root = src                                              # pointer jumping: reach doubles per step
    while True:
        nxt = root.gather(1, root)
        if torch.equal(nxt, root):
            break
        root = nxt
    tokens = fresh.gather(1, root).to(torch.int32).contiguous()
    lengths = (L // 2 + torch.randint(0, L - L // 2 + 1, (B,), generator=g, device=device)).to(torch.int32)
    return tokens, lengths


@dataclass(frozen=True)
class Eagle2Workload:
    name: str
    B: int
    V: int
    dtype: str
    T: float
    k: int               # candidates per frontier node = nodes expanded per step
    depth: int           # expansion steps
    m: int               # nodes kept by the rerank beside the root
    sigma: float = 3.0
    data_seed: int = 3000

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def M(self) -> int:
        """Nodes of a fully grown tree: the root, k at the first step, k*k after."""
        return 1 + self.k + (self.depth - 1) * self.k * self.k

    def frontier_size(self, step: int) -> int:
        return 1 if step == 0 else self.k

    def offset(self, step: int) -> int:
        return 1 if step == 0 else 1 + self.k + (step - 1) * self.k * self.k


EAGLE2_WORKLOADS = {
    # the node budget of the static tree workload (63 nodes, depth 5) spent
    # dynamically: 8 candidates per node, 8 nodes grown per step
    "eg1": Eagle2Workload("eg1", B=32, V=128256, dtype="bf16", T=1.0, k=8, depth=5, m=62, data_seed=3001),
}

_MASK63 = (1 << 63) - 1


def _mix64(x: int) -> int:
    """splitmix64 finaliser (Steele, Lea and Flood, OOPSLA 2014), 63 bits out."""
    x &= (1 << 64) - 1
    x = (x + 0x9E3779B97F4A7C15) & ((1 << 64) - 1)
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & ((1 << 64) - 1)
    return (x ^ (x >> 31)) & _MASK63


def root_key(w: Eagle2Workload, b: int) -> int:
    return _mix64(w.data_seed * 1000003 + b)


def node_key(parent_key: int, token: int) -> int:
    return _mix64(parent_key * 31 + token + 1)


def draft_rows(w: Eagle2Workload, keys, device="cpu"):
    """The stand-in draft's logits at the nodes with these path keys: [len(keys), V]."""
    out = torch.empty((len(keys), w.V), dtype=torch.float32)
    g = torch.Generator(device="cpu")
    for i, key in enumerate(keys):
        g.manual_seed(int(key))
        out[i] = torch.randn(w.V, generator=g) * w.sigma
    return out.to(w.torch_dtype).to(device)


def eagle2_step_rows(w: Eagle2Workload, step: int, device="cpu"):
    """Per-step draft rows [B, F, V] for timing (fresh seeded noise; the row
    of a frontier slot does not follow a path)."""
    g = _gen(device, w.data_seed + 7 * step + 1)
    F = w.frontier_size(step)
    return (torch.randn((w.B, F, w.V), generator=g, device=device) * w.sigma).to(w.torch_dtype)
