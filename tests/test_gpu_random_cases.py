"""Randomised parity cases: every verification kind, the drafter and the
top-k on seeded random shapes (odd vocabularies, empty drafts, one-node and
random trees), both element types, temperatures including 0, ties, masked
counts, and inputs one element past a 16-byte boundary (the plain-load path),
each against the oracle with the parity rule of the other tests: bit-exact
except sequences the oracle flags near a decision or CDF boundary."""
import random

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import NTHREADS, compare_chain, record_parity
from sampling_row_online_gb300 import binding

pytestmark = pytest.mark.gpu

VS = [1, 2, 7, 8, 9, 31, 33, 100, 1000, 4095, 4096, 4097, 8191, 16385, 32000, 50257]


def place(t, unaligned):
    """t's values in a fresh contiguous tensor, one element past a 16-byte boundary if unaligned."""
    n = t.numel()
    if unaligned:
        buf = torch.empty(n + 1, dtype=t.dtype, device="cuda")
        out = buf[1:1 + n].view(t.shape)
    else:
        out = torch.empty(t.shape, dtype=t.dtype, device="cuda")
    out.copy_(t)
    return out


def chain_case(i, rng):
    B, K = rng.randint(1, 40), rng.randint(0, 8)
    V = rng.choice(VS + [rng.randint(1, 70000)])
    tdt = rng.choice([torch.float32, torch.bfloat16])
    T = rng.choice([0.0, 0.5, 0.7, 1.0, 1.3])
    un = rng.random() < 0.3
    sd = rng.choice([0.05, 1.0, 3.0])
    g = torch.Generator(device="cuda").manual_seed(1000 + i)
    zt32 = torch.randn((B, K + 1, V), generator=g, device="cuda") * 3
    zd32 = zt32[:, :K] + torch.randn((B, K, V), generator=g, device="cuda") * sd
    good = torch.rand((B, K), generator=g, device="cuda") < 0.6
    x = torch.where(good, zd32.argmax(-1), torch.randint(0, V, (B, K), generator=g, device="cuda")).to(torch.int32)
    zt, zd = place(zt32.to(tdt), un), place(zd32.to(tdt), un)
    seed = rng.randint(0, 2 ** 40)
    out, n = binding.spec_verify(zt, zd if T > 0 else None, x.contiguous(), T, seed)
    st = binding.spec_get_status()
    assert st == 0, f"status {st}"
    ref = oracle.verify_chain(zt.cpu(), zd.cpu() if T > 0 else None, x.cpu(), T, seed, nthreads=NTHREADS)
    compare_chain(out.cpu().numpy(), n.cpu().numpy(), ref, positions=B * max(K, 1), kind="random-chain")
    return f"chain B={B} K={K} V={V} {tdt} T={T} unaligned={un}"


def tree_case(i, rng):
    B, N = rng.randint(1, 20), rng.randint(1, 100)
    V = rng.choice(VS + [rng.randint(1, 70000)])
    tdt = rng.choice([torch.float32, torch.bfloat16])
    un = rng.random() < 0.3
    parent = [-1] + [rng.randint(0, c - 1) for c in range(1, N)]
    g = torch.Generator(device="cuda").manual_seed(2000 + i)
    z32 = torch.randn((B, N, V), generator=g, device="cuda") * 3
    if rng.random() < 0.3:
        z32 = torch.round(z32)          # many ties
    zt = place(z32.to(tdt), un)
    top = zt.float().argmax(-1).to(torch.int32)
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    tok = torch.where(torch.rand((B, N), generator=g, device="cuda") < 0.6, top[:, par.clamp(min=0).long()],
                      torch.randint(0, V, (B, N), generator=g, device="cuda").to(torch.int32)).to(torch.int32)
    path, ln = binding.spec_verify_tree_greedy(zt, par, tok.contiguous())
    assert binding.spec_get_status() == 0
    rp, rl, _ = oracle.verify_tree_greedy(zt.cpu(), par.cpu(), tok.cpu(), nthreads=NTHREADS)
    assert np.array_equal(ln.cpu().numpy(), rl), "length"
    assert np.array_equal(path.cpu().numpy(), rp), "path"
    return f"tree B={B} N={N} V={V} {tdt} unaligned={un}"


def topk_case(i, rng):
    R = rng.randint(1, 300)
    V = rng.choice([v for v in VS if v >= 32] + [rng.randint(32, 70000)])
    k = rng.randint(1, 32)
    tdt = rng.choice([torch.float32, torch.bfloat16])
    T = rng.choice([0.5, 1.0, 1.7])
    un = rng.random() < 0.3
    g = torch.Generator(device="cuda").manual_seed(3000 + i)
    z32 = torch.randn((R, V), generator=g, device="cuda") * 3
    if rng.random() < 0.3:
        z32 = torch.round(z32 * 2) / 2  # ties
    z = place(z32.to(tdt), un)
    tok, prob = binding.spec_topk(z, k, T)
    assert binding.spec_get_status() == 0
    rt, rp = oracle.topk_prob(z.cpu(), k, T)
    assert np.array_equal(tok.cpu().numpy(), rt), "tokens"
    np.testing.assert_allclose(prob.cpu().numpy(), rp, rtol=2e-5, atol=1e-30)
    return f"topk R={R} V={V} k={k} {tdt} T={T} unaligned={un}"


def tree_sample_case(i, rng):
    B, N = rng.randint(1, 16), rng.randint(1, 64)
    V = rng.choice(VS + [rng.randint(1, 70000)])
    tdt = rng.choice([torch.float32, torch.bfloat16])
    T = rng.choice([0.5, 0.8, 1.0, 1.3])
    un = rng.random() < 0.3
    parent = [-1] + [rng.randint(0, c - 1) for c in range(1, N)]
    g = torch.Generator(device="cuda").manual_seed(4000 + i)
    zt32 = torch.randn((B, N, V), generator=g, device="cuda") * 3
    zd32 = zt32 + torch.randn((B, N, V), generator=g, device="cuda") * rng.choice([0.1, 1.0, 3.0])
    zt, zd = place(zt32.to(tdt), un), place(zd32.to(tdt), un)
    par = torch.tensor(parent, dtype=torch.int32, device="cuda")
    top = zd.float().argmax(-1).to(torch.int32)
    tok = torch.where(torch.rand((B, N), generator=g, device="cuda") < 0.6, top[:, par.clamp(min=0).long()],
                      torch.randint(0, V, (B, N), generator=g, device="cuda").to(torch.int32)).to(torch.int32)
    per_seq = rng.random() < 0.4
    pars = par.unsqueeze(0).expand(B, -1).contiguous() if per_seq else par
    seed = rng.randint(0, 2 ** 40)
    path, ln = binding.spec_verify_tree(zt, zd, pars, tok.contiguous(), T, seed)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_tree_sample(zt.cpu(), zd.cpu(), par.cpu(), tok.cpu(), T, seed, nthreads=NTHREADS)
    ok = (ln.cpu().numpy() == ref["length"]) & np.all(path.cpu().numpy() == ref["path"], axis=1)
    record_parity("random-tree_sample", ok, ref["near"], B * max(1, N - 1), "(trees)")
    return f"tree_sample B={B} N={N} V={V}"


def points_case(i, rng):
    B, K = rng.randint(1, 40), rng.randint(0, 8)
    V = rng.choice(VS + [rng.randint(1, 70000)])
    tdt = rng.choice([torch.float32, torch.bfloat16])
    T = rng.choice([0.0, 0.7, 1.0, 1.3])
    un = rng.random() < 0.3
    g = torch.Generator(device="cuda").manual_seed(5000 + i)
    zt32 = torch.randn((B, K + 1, V), generator=g, device="cuda") * 3
    zt = place(zt32.to(tdt), un)
    top = zt32[:, :K].argmax(-1).to(torch.int32)
    x = torch.where(torch.rand((B, K), generator=g, device="cuda") < 0.6, top,
                    torch.randint(0, V, (B, K), generator=g, device="cuda").to(torch.int32)).to(torch.int32)
    counts = None
    if rng.random() < 0.5:
        counts = torch.randint(0, K + 1, (B,), generator=g, device="cuda").to(torch.int32)
        x = torch.where(torch.arange(K, device="cuda")[None, :] < counts[:, None], x, -1).to(torch.int32)
    seed = rng.randint(0, 2 ** 40)
    out, n = binding.spec_verify_points(zt, x.contiguous(), T, seed, draft_counts=counts)
    assert binding.spec_get_status() == 0
    ref = oracle.verify_points(zt.cpu(), x.cpu(), None if counts is None else counts.cpu(), T, seed,
                               nthreads=NTHREADS)
    ok = (n.cpu().numpy() == ref["n"]) & np.all(out.cpu().numpy() == ref["tokens"], axis=1)
    record_parity("random-points", ok, ref["near"], B * max(K, 1))
    return f"points B={B} K={K} V={V}"


def ngram_case(i, rng):
    B, L = rng.randint(1, 32), rng.randint(1, 20000)
    n_min = rng.randint(1, 4)
    n_max = rng.randint(n_min, min(64, n_min + rng.choice([0, 3, 7, 12])))
    K, hits = rng.randint(1, 8), rng.choice([1, 1, 2, 3])
    g = torch.Generator(device="cuda").manual_seed(6000 + i)
    vocab = rng.choice([2, 5, 50, 32000])
    tokens = torch.randint(0, vocab, (B, L), generator=g, device="cuda").to(torch.int32)
    lengths = torch.randint(0, L + 1, (B,), generator=g, device="cuda").to(torch.int32)
    d, c = binding.spec_ngram_propose(tokens, lengths, n_min, n_max, K, min_hits=hits)
    assert binding.spec_get_status() == 0
    rd, rc = oracle.ngram_propose(tokens.cpu().numpy(), lengths.cpu().numpy(), n_min, n_max, K, min_hits=hits)
    assert np.array_equal(c.cpu().numpy(), rc), "counts"
    assert np.array_equal(d.cpu().numpy(), rd), "drafts"
    return f"ngram B={B} L={L} n={n_min}..{n_max} K={K} hits={hits} vocab={vocab}"



KINDS = {"chain": chain_case, "tree": tree_case, "topk": topk_case, "tree_sample": tree_sample_case,
         "points": points_case, "ngram": ngram_case}


@pytest.mark.parametrize("i", range(20))
@pytest.mark.parametrize("kind", sorted(KINDS))
def test_random_case(kind, i):
    rng = random.Random(f"{kind}-{i}")
    desc = KINDS[kind](i, rng)
    assert desc
