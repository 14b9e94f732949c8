// EAGLE-2 tree budget (infra-guide, "5.3 Medusa, EAGLE và MTP", §5.1-§5.3):
// the draft's confidence steers a limited node budget; a node's value is the
// product of the confidences on its path; an expansion phase grows the best
// nodes, a rerank keeps the best nodes of all for verification.
//
//   topk_kernel    per draft row: the k most probable tokens (ties to the
//                  lower index) and their probabilities softmax(z / T)
//   expand_kernel  per tree: candidate value = parent value x probability,
//                  the next frontier = the k_next best new candidates
//   rerank_kernel  per tree: the root and the m best nodes (value, then
//                  smaller depth, then lower id), listed by depth, parents
//                  remapped to list positions
#pragma once

#include <cstdint>

#include "kernels.cuh"

namespace spec {

constexpr int TOPK_MAX = 32;           // largest k of a top-k row
constexpr int EAGLE_MAX_CAND = 4096;   // largest F * k of one expansion step
constexpr int EAGLE_MAX_NODES = 8192;  // largest M of a rerank

// Order-preserving map of a float to 32 bits (larger float, larger key);
// -inf maps below every finite value, and -0 is taken as +0 (they compare
// equal, so they must tie).
__device__ __forceinline__ uint32_t float_order(float x) {
  uint32_t b = __float_as_uint(x);
  b = b == 0x80000000u ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_float(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
// (logit, index) key: larger logit first, ties to the lower index.  0 is
// below every real key (an empty slot).
__device__ __forceinline__ unsigned long long topk_key(float x, int i) {
  return (static_cast<unsigned long long>(float_order(x)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(i));
}

// Sorted (descending) register list of KMAX keys of which the last k are
// live: the first KMAX - k slots hold a sentinel above every key, which no
// insertion displaces, so the k-th live key is always key[KMAX - 1] and no
// slot is ever indexed with a run-time value (the list stays in registers).
constexpr unsigned long long TOPK_SENTINEL = ~0ull;

template <int KMAX>
struct TopList {
  unsigned long long key[KMAX];
  __device__ __forceinline__ void clear(int k) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) key[j] = j < KMAX - k ? TOPK_SENTINEL : 0ull;
  }
  // Inserts c (bubbling the displaced keys down); the last key drops out.
  __device__ __forceinline__ void insert(unsigned long long c) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const unsigned long long cur = key[j];
      const bool sw = c > cur;
      key[j] = sw ? c : cur;
      c = sw ? cur : c;
    }
  }
  __device__ __forceinline__ unsigned long long last() const { return key[KMAX - 1]; }
  // The largest live key (0 if none is left).
  __device__ __forceinline__ unsigned long long head() const {
    unsigned long long h = 0ull;
#pragma unroll
    for (int j = KMAX - 1; j >= 0; --j) h = key[j] != TOPK_SENTINEL ? key[j] : h;
    return h;
  }
  // Retires key h (it becomes a sentinel).
  __device__ __forceinline__ void retire(unsigned long long h) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) key[j] = key[j] == h ? TOPK_SENTINEL : key[j];
  }
};

__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

struct TopkParams {
  const void *z;          // [R, V] logits (row r at z + r * V)
  int R, V, k;
  float c;                // log2(e) / T
  int32_t *out_tok;       // [R, k] or node_tok (see dst_* below)
  float *out_prob;        // [R, k] or node_val
  // expansion layout: row r = (b, f) writes its k results to node slots
  // offset + f * k + j of tree b (arrays of stride cap), parent frontier[b, f]
  int F, cap, offset;     // F == 0: plain [R, k] outputs
  const int32_t *frontier;
  int32_t *node_par;
  int32_t *status;
};

struct TopkShared {
  unsigned long long wk[NWARP][TOPK_MAX];  // per-warp merged lists
  float wm[NWARP], ws[NWARP];
  float m, s;
};

// Online (max, sum of 2^((x - max) c)) update with one value.
__device__ __forceinline__ void topk_online(float x, float c, float &m, float &s) {
  if (x > m) {
    s = s * ex2((m - x) * c) + 1.f;  // m = -inf: ex2(-inf) = 0
    m = x;
  } else if (x != -INFINITY) {
    s += ex2(fmaf(x, c, -m * c));
  }
}

// Offers (x, i) to a thread's list; kkey / thr track its k-th key and logit.
template <int KMAX>
__device__ __forceinline__ void topk_offer(TopList<KMAX> &L, unsigned long long &kkey, float &thr,
                                           float x, int i) {
  if (x >= thr) {
    const unsigned long long key = topk_key(x, i);
    if (key > kkey) {
      L.insert(key);
      kkey = L.last();
      thr = kkey ? order_float(static_cast<uint32_t>(kkey >> 32)) : -INFINITY;
    }
  }
}

constexpr int TOPK_U = 8;  // 16-byte loads in flight per thread

template <int DT, bool VEC, int KMAX>
__global__ void __launch_bounds__(NT, KMAX <= 16 ? 2 : 1) topk_kernel(TopkParams p) {
  __shared__ TopkShared sh;
  constexpr int VE = Elem<DT>::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int k = p.k;
  pdl_launch_dependents();
  pdl_wait();
  const unsigned char *row = static_cast<const unsigned char *>(p.z) +
                             static_cast<size_t>(r) * p.V * Elem<DT>::BYTES;
  TopList<KMAX> L;
  L.clear(k);
  float thr = -INFINITY;            // logit of the k-th kept key (-inf while slots are empty)
  unsigned long long kkey = 0ull;    // the k-th kept key
  float m = -INFINITY, s = 0.f;
  if (VEC) {
    // 16-byte vectors, TOPK_U per thread in flight; a thread's indices increase
    const int nvec = p.V / VE;
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    for (int base = tid; base < nvec; base += TOPK_U * NT) {
      uint4 q[TOPK_U];
#pragma unroll
      for (int u = 0; u < TOPK_U; ++u) {
        const int vi = base + u * NT;
        q[u] = vi < nvec ? __ldg(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < TOPK_U; ++u) {
        const int vi = base + u * NT;
        if (vi < nvec) {
          float f[VE];
          Elem<DT>::unpack(q[u], f);
          float vm = f[0];
#pragma unroll
          for (int e = 1; e < VE; ++e) vm = fmaxf(vm, f[e]);
          if (vm > m) {
            s *= ex2((m - vm) * p.c);
            m = vm;
          }
          if (m != -INFINITY) {
            const float mc = m * p.c;
#pragma unroll
            for (int e = 0; e < VE; ++e) s += ex2(fmaf(f[e], p.c, -mc));
          }
          if (vm >= thr) {
#pragma unroll
            for (int e = 0; e < VE; ++e) topk_offer(L, kkey, thr, f[e], vi * VE + e);
          }
        }
      }
    }
  } else {
    for (int i = tid; i < p.V; i += NT) {
      const float x = Elem<DT>::load(row, i);
      topk_online(x, p.c, m, s);
      topk_offer(L, kkey, thr, x, i);
    }
  }

  // row normalisers: warp, then CTA
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float mn = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * ex2((m - mn) * p.c)) + (m2 == -INFINITY ? 0.f : s2 * ex2((m2 - mn) * p.c));
    m = mn;
  }
  // warp top-k: k rounds, the lane holding the best head pops it
  for (int j = 0; j < k; ++j) {
    const unsigned long long h = L.head();
    const unsigned long long best = warp_max_key(h);
    if (lane == 0) sh.wk[warp][j] = best;
    if (h == best && best != 0ull) L.retire(best);
  }
  if (lane == 0) {
    sh.wm[warp] = m;
    sh.ws[warp] = s;
  }
  __syncthreads();
  if (warp != 0) return;
  // CTA: lanes 0..NWARP-1 hold the warp lists (shared memory heads)
  m = lane < NWARP ? sh.wm[lane] : -INFINITY;
  s = lane < NWARP ? sh.ws[lane] : 0.f;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float mn = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * ex2((m - mn) * p.c)) + (m2 == -INFINITY ? 0.f : s2 * ex2((m2 - mn) * p.c));
    m = mn;
  }
  int head = 0;
  for (int j = 0; j < k; ++j) {
    const unsigned long long mine = lane < NWARP && head < k ? sh.wk[lane][head] : 0ull;
    const unsigned long long best = warp_max_key(mine);
    if (mine == best && best != 0ull) ++head;
    if (lane == 0) {
      const int i = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best));
      const float x = order_float(static_cast<uint32_t>(best >> 32));
      const float prob = ex2(fmaf(x, p.c, -m * p.c)) / s;
      if (p.F == 0) {
        p.out_tok[static_cast<size_t>(r) * k + j] = i;
        p.out_prob[static_cast<size_t>(r) * k + j] = prob;
      } else {
        const int b = r / p.F, f = r - b * p.F;
        const size_t slot = static_cast<size_t>(b) * p.cap + p.offset + f * k + j;
        p.out_tok[slot] = i;
        p.out_prob[slot] = prob;  // the select step multiplies by the parent's value
        p.node_par[slot] = __ldg(p.frontier + r);
      }
    }
  }
}

struct EagleParams {
  int B, F, k, cap, offset, k_next;  // expansion step
  int M, m;                          // rerank
  const int32_t *frontier;           // [B, F]
  int32_t *node_tok;                 // [B, cap] (rerank: [B, M])
  float *node_val;
  int32_t *node_par;
  int32_t *out_next;                 // [B, k_next] next frontier (node ids)
  int32_t *out_par, *out_tok, *out_idx;  // [B, m + 1] the kept tree
  int32_t *status;
};

// Expansion step, second half (one CTA per tree): the top-k kernel has put
// each candidate's probability, token and parent in its node slot; here the
// value becomes parent value x probability and the k_next best candidates
// (value, ties to the lower id) become the next frontier, best first.
__global__ void __launch_bounds__(NT) expand_select_kernel(EagleParams p) {
  __shared__ unsigned long long key[EAGLE_MAX_CAND];
  __shared__ int bad;
  const int tid = threadIdx.x, b = blockIdx.x;
  const int n = p.F * p.k;
  pdl_launch_dependents();
  if (tid == 0) bad = 0;
  pdl_wait();
  __syncthreads();
  float *val = p.node_val + static_cast<size_t>(b) * p.cap;
  const int32_t *par = p.node_par + static_cast<size_t>(b) * p.cap;
  for (int i = tid; i < n; i += NT) {
    const int c = p.offset + i;
    const int u = par[c];
    if (u < 0 || u >= p.offset) {  // a frontier id outside the tree so far
      atomicOr(&bad, 1);
      key[i] = 0ull;
      continue;
    }
    const float v = __fmul_rn(val[u], val[c]);
    val[c] = v;
    key[i] = (static_cast<unsigned long long>(float_order(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(i));
  }
  __syncthreads();
  int32_t *next = p.out_next + static_cast<size_t>(b) * p.k_next;
  if (bad) {
    for (int j = tid; j < p.k_next; j += NT) next[j] = -1;
    if (tid == 0) atomicOr(p.status, ST_PARENT);
    return;
  }
  for (int i = tid; i < n; i += NT) {
    const unsigned long long mine = key[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += key[j] > mine;
    if (rank < p.k_next) next[rank] = p.offset + i;
  }
}

// Rerank (one CTA per tree of M nodes): keep the root and the m best other
// nodes by (value, then smaller depth, then lower id); list them by depth,
// then rank; parents become list positions.  Dynamic shared memory: key[M]
// (8 B), depth[M], rank[M] (4 B each), byrank[m].
__global__ void __launch_bounds__(NT) rerank_kernel(EagleParams p) {
  extern __shared__ __align__(128) unsigned char rerank_smem[];
  unsigned long long *key = reinterpret_cast<unsigned long long *>(rerank_smem);
  int *depth = reinterpret_cast<int *>(key + p.M);
  int *rank = depth + p.M;
  int *byrank = rank + p.M;
  __shared__ int bad;
  const int tid = threadIdx.x, b = blockIdx.x;
  const int M = p.M, m = p.m;
  pdl_launch_dependents();
  if (tid == 0) bad = 0;
  pdl_wait();
  __syncthreads();
  const float *val = p.node_val + static_cast<size_t>(b) * M;
  const int32_t *par = p.node_par + static_cast<size_t>(b) * M;
  const int32_t *tok = p.node_tok + static_cast<size_t>(b) * M;
  for (int c = tid; c < M; c += NT) {
    const int u = __ldg(par + c);
    if (c == 0 ? u != -1 : (u < 0 || u >= c)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (!bad) {
    for (int c = tid; c < M; c += NT) {  // parent[c] < c: the walk ends at the root
      int d = 0;
      for (int u = c; u != 0; u = __ldg(par + u)) ++d;
      depth[c] = d;
    }
    __syncthreads();
    for (int c = tid; c < M; c += NT)
      key[c] = c == 0 ? 0ull
                      : (static_cast<unsigned long long>(float_order(__ldg(val + c))) << 32) |
                            (static_cast<unsigned long long>(255 - min(depth[c], 255)) << 24) |
                            (0xFFFFFFu - static_cast<uint32_t>(c));
    __syncthreads();
    for (int c = tid; c < M; c += NT) {
      int r = -1;
      if (c > 0) {
        const unsigned long long mine = key[c];
        r = 0;
        for (int j = 1; j < M; ++j) r += key[j] > mine;
        if (r < m) byrank[r] = c;
      }
      rank[c] = r;
    }
    __syncthreads();
    for (int r = tid; r < m; r += NT) {  // a kept node's parent must be kept
      const int u = __ldg(par + byrank[r]);
      if (u != 0 && rank[u] >= m) atomicOr(&bad, 1);
    }
    __syncthreads();
  }
  int32_t *op = p.out_par + static_cast<size_t>(b) * (m + 1);
  int32_t *ot = p.out_tok + static_cast<size_t>(b) * (m + 1);
  int32_t *oi = p.out_idx + static_cast<size_t>(b) * (m + 1);
  if (bad) {
    for (int i = tid; i <= m; i += NT) op[i] = ot[i] = oi[i] = -1;
    if (tid == 0) atomicOr(p.status, ST_PARENT);
    return;
  }
  // list position of the kept node of rank r: 1 + kept nodes before it by
  // (depth, rank); written to rank[] of that node for the parent remap
  __syncthreads();
  for (int r = tid; r < m; r += NT) {
    const int c = byrank[r], d = depth[c];
    int q = 1;
    for (int r2 = 0; r2 < m; ++r2) {
      const int d2 = depth[byrank[r2]];
      q += d2 < d || (d2 == d && r2 < r);
    }
    key[c] = static_cast<unsigned long long>(q);  // key[] reused: list position
  }
  __syncthreads();
  if (tid == 0) {
    op[0] = -1;
    ot[0] = __ldg(tok);
    oi[0] = 0;
  }
  for (int r = tid; r < m; r += NT) {
    const int c = byrank[r];
    const int q = static_cast<int>(key[c]);
    const int u = __ldg(par + c);
    op[q] = u == 0 ? 0 : static_cast<int>(key[u]);
    ot[q] = __ldg(tok + c);
    oi[q] = c;
  }
}

}  // namespace spec
