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

// A warp's sorted (descending) list of its k best keys, k <= 32, one key per
// lane: lane j holds the j-th best (0 in unused or not yet filled slots).
// Inserting a key is one shuffle and a select per lane; the k-th key (lane
// k - 1) is the warp's admission threshold.
__device__ __forceinline__ unsigned long long warp_list_insert(unsigned long long lk, unsigned long long cand,
                                                               int lane) {
  const unsigned long long up = __shfl_up_sync(0xFFFFFFFFu, lk, 1);
  return lk > cand ? lk : ((lane == 0 || up > cand) ? cand : up);
}

// Sorts one float per lane across the warp, largest in lane 0 (bitonic).
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
      const bool up = (lane & size) == 0;        // this block sorts descending
      const bool low = (lane & stride) == 0;     // the lower lane of the pair
      v = (low == up) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

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
  unsigned long long *timer;  // measurement (or null): [0] earliest CTA start, [1] latest CTA end,
                              // [2] latest row written (global-timer ns)
};

__device__ __forceinline__ void topk_stamp(const TopkParams &p, int k, bool first) {
  if (!p.timer) return;
  const unsigned long long t = clock_ns();
  if (first)
    atomicMin(p.timer + k, t);
  else
    atomicMax(p.timer + k, t);
}

constexpr int TOPK_MAX_CLUSTER = 8;  // CTAs sharing one row
constexpr int TOPK_NT = 512;         // threads of a top-k CTA
constexpr int TOPK_NWARP = TOPK_NT / 32;
constexpr int TOPK_GS = TOPK_NT / 32;  // threads per group of the threshold (32 groups)
static_assert(TOPK_GS <= 32 && 32 % TOPK_GS == 0, "threshold groups lie within a warp");
constexpr int TOPK_BUF = 1024;       // candidate keys a CTA collects before falling back

struct TopkShared {
  unsigned long long buf[TOPK_BUF];                   // candidates (keys >= the threshold)
  uint4 pv[TOPK_NT];                                       // each thread's best vector, fetched again
  float gmax[32];                                     // maxima of the threshold's groups
  int nbuf;
  unsigned long long wk[TOPK_NWARP][TOPK_MAX];             // per-warp lists (fallback path)
  unsigned long long ctak[TOPK_MAX];                  // this CTA's top k
  unsigned long long ck[TOPK_MAX_CLUSTER][TOPK_MAX];  // rank 0: the CTA lists of the cluster
  float wm[TOPK_NWARP], ws[TOPK_NWARP];
  float cm[TOPK_MAX_CLUSTER], cs[TOPK_MAX_CLUSTER];   // rank 0: the CTA normalisers
  unsigned long long bar_key;                         // largest k-th key of any warp so far
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

// 16-byte loads per thread per round; pass 1 issues the next round's loads
// before it weighs the current one, so up to 2 * TOPK_U are in flight
constexpr int TOPK_U = 4;

// Element e (0 <= e < VE, a run-time value) of a packed 16-byte vector.
template <int DT>
__device__ __forceinline__ float elem_of(const uint4 &q, int e) {
  if (DT == 0) {
    const uint32_t w = e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
    return __uint_as_float(w);
  }
  const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Warp-wide admission: lanes with candidates (bit e of cm: element e of
// their vector q, at index base_i + e) insert them one at a time, the lowest
// lane first; after each insert every lane drops the candidates that no
// longer beat the bar.  The bar is the largest k-th key of any warp of the
// CTA (shared in *bar): the CTA's k-th key is at least that, so no key below
// it can reach the CTA's top k.  Uniform control flow.
template <int DT>
__device__ __forceinline__ void warp_admit(uint32_t cm, const uint4 &q, int base_i, int k, int lane,
                                           unsigned long long &lk, unsigned long long &kkey, float &thr,
                                           unsigned long long *bar) {
  constexpr int VE = Elem<DT>::VE;
  unsigned ballot = __ballot_sync(0xFFFFFFFFu, cm != 0u);
  while (ballot) {
    const int src = __ffs(ballot) - 1;
    unsigned long long key = 0ull;
    if (lane == src) {
      const int e = __ffs(cm) - 1;
      cm &= cm - 1u;
      key = topk_key(elem_of<DT>(q, e), base_i + e);
    }
    key = __shfl_sync(0xFFFFFFFFu, key, src);
    if (key > kkey) {  // uniform
      lk = warp_list_insert(lk, key, lane);
      const unsigned long long own = __shfl_sync(0xFFFFFFFFu, lk, k - 1);
      unsigned long long b = 0ull;
      if (lane == 0) b = own ? atomicMax(bar, own) : *reinterpret_cast<volatile unsigned long long *>(bar);
      b = __shfl_sync(0xFFFFFFFFu, b, 0);
      kkey = own > b ? own : b;
      thr = kkey ? order_float(static_cast<uint32_t>(kkey >> 32)) : -INFINITY;
#pragma unroll
      for (int e = 0; e < VE; ++e)
        if ((cm >> e) & 1u)
          if (elem_of<DT>(q, e) < thr) cm &= ~(1u << e);
    }
    ballot = __ballot_sync(0xFFFFFFFFu, cm != 0u);
  }
}

// The k best keys of this CTA's slice (vectors [lo, hi) for VEC, else
// elements [lo, hi)) by lockstep admission: the fallback when too many
// elements tie at the threshold (flat or masked rows).  Leaves them in
// sh.ctak[0 .. k-1].
template <int DT, bool VEC>
__device__ void topk_slice_by_admission(const unsigned char *row, int lo, int hi, int k, TopkShared &sh) {
  constexpr int VE = Elem<DT>::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh.bar_key = 0ull;
  __syncthreads();
  unsigned long long lk = 0ull, kkey = 0ull;
  float thr = -INFINITY;
  if (VEC) {
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    for (int base = lo + warp * 32; base < hi; base += TOPK_NT) {  // warp-uniform
      const int vi = base + lane;
      const uint4 q = vi < hi ? __ldg(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t cm = 0u;
      if (vi < hi) {
        float f[VE];
        Elem<DT>::unpack(q, f);
#pragma unroll
        for (int e = 0; e < VE; ++e) cm |= (f[e] >= thr ? 1u : 0u) << e;
      }
      warp_admit<DT>(cm, q, vi * VE, k, lane, lk, kkey, thr, &sh.bar_key);
    }
  } else {
    for (int i0 = lo + warp * 32; i0 < hi; i0 += TOPK_NT) {  // warp-uniform
      const int i = i0 + lane;
      const float x = i < hi ? Elem<DT>::load(row, i) : -INFINITY;
      const uint4 q = make_uint4(__float_as_uint(x), 0u, 0u, 0u);
      warp_admit<0>((i < hi && x >= thr) ? 1u : 0u, q, i, k, lane, lk, kkey, thr, &sh.bar_key);
    }
  }
  if (lane < k) sh.wk[warp][lane] = lk;
  __syncthreads();
  if (warp == 0) {
    int head = 0;
    for (int j = 0; j < k; ++j) {
      const unsigned long long mine = lane < TOPK_NWARP && head < k ? sh.wk[lane][head] : 0ull;
      const unsigned long long best = warp_max_key(mine);
      if (mine == best && best != 0ull) ++head;
      if (lane == 0) sh.ctak[j] = best;
    }
  }
  __syncthreads();
}

// (max, sum of 2^((z - max) c)) of the states held by lanes 0 .. n-1 (n a
// power of two up to 32), into every one of those lanes: the maximum first,
// then one rescale per lane and the sum, so the dependent chain holds one
// exponential.
__device__ __forceinline__ void group_ms(float &m, float &s, float c, int n) {
  float M = m;
  for (int o = 1; o < n; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  float t = (M == -INFINITY || m == -INFINITY) ? 0.f : s * ex2((m - M) * c);
  for (int o = 1; o < n; o <<= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  m = M;
  s = t;
}

// Rank 0 of a row's cluster, one warp: merges the G CTA lists (each sorted,
// best first; keys distinct, empty slots 0), combines the G slice
// normalisers, and writes the row's k tokens and probabilities (the
// expansion layout writes straight into the node arrays).  `poisoned`: a
// wait of the row ran out; the row is written as tokens -1 with probability
// 0 (parents -1).
__device__ __forceinline__ void topk_write_row(const TopkParams &p, int r, int G, int k,
                                               const unsigned long long (*ck)[TOPK_MAX], const float *cm,
                                               const float *cs, int lane, bool poisoned) {
  float m = lane < G ? cm[lane] : -INFINITY;
  float s = lane < G ? cs[lane] : 0.f;
  group_ms(m, s, p.c, G);
  m = __shfl_sync(0xFFFFFFFFu, m, 0);
  const float inv_s = 1.f / __shfl_sync(0xFFFFFFFFu, s, 0);
  auto put = [&](int j, int idx, float prob, int par) {
    if (p.F == 0) {
      p.out_tok[static_cast<size_t>(r) * k + j] = idx;
      p.out_prob[static_cast<size_t>(r) * k + j] = prob;
    } else {
      const int b = r / p.F, f = r - b * p.F;
      const size_t slot = static_cast<size_t>(b) * p.cap + p.offset + f * k + j;
      p.out_tok[slot] = idx;
      p.out_prob[slot] = prob;  // the select step multiplies by the parent's value
      p.node_par[slot] = par;
    }
  };
  if (poisoned) {
    for (int j = lane; j < k; j += 32) put(j, -1, 0.f, -1);
    return;
  }
  // slot (g, j) of the lists: its rank is j plus the keys above it in the
  // other lists; the k best are written in parallel
  for (int l = lane; l < G * k; l += 32) {
    const int g = l / k, j = l - g * k;
    const unsigned long long key = ck[g][j];
    if (key == 0ull) continue;
    int rk = j;
    for (int g2 = 0; g2 < G; ++g2) {
      if (g2 == g) continue;
#pragma unroll
      for (int j2 = 0; j2 < TOPK_MAX; ++j2) rk += j2 < k && ck[g2][j2] > key;
    }
    if (rk < k) {
      const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
      const float x = order_float(static_cast<uint32_t>(key >> 32));
      put(rk, idx, ex2(fmaf(x, p.c, -m * p.c)) * inv_s, p.F == 0 ? 0 : __ldg(p.frontier + r));
    }
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(TOPK_NT, 2) topk_kernel(TopkParams p) {
  __shared__ TopkShared sh;
  constexpr int VE = Elem<DT>::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = static_cast<int>(cluster_size());  // CTAs per row, each a contiguous slice
  const int rank = static_cast<int>(cluster_rank());
  const int r = blockIdx.x / G;
  const int k = p.k;
  pdl_launch_dependents();
  if (tid == 0) sh.nbuf = 0;
  pdl_wait();
  if (tid == 0) topk_stamp(p, 0, true);
  const unsigned char *row = static_cast<const unsigned char *>(p.z) +
                             static_cast<size_t>(r) * p.V * Elem<DT>::BYTES;
  const int n = VEC ? p.V / VE : p.V;  // vectors (VEC) or elements
  const int per = (n + G - 1) / G;
  const int lo = min(n, rank * per), hi = min(n, lo + per);

  // pass 1: online (max, sum) and the thread's own largest logit; with
  // vector loads, also the index of the thread's best vector (the first to
  // reach the maximum; -1: no vector with a finite maximum) and the largest
  // maximum of its other vectors
  float m = -INFINITY, s = 0.f, tmax = -INFINITY;
  float vm2 = -INFINITY;
  int j1 = -1;
  if (VEC) {
    // the streaming kernel's per-vector update (packed maxima, paired sums);
    // the online state's maximum is the thread's own largest logit
    Online st;  // st.m is also the best vector's maximum
    st.init();
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    // thread (warp, lane) reads vectors lo + warp * 32 + lane + j * TOPK_NT
    auto fetch = [&](uint4 (&d)[TOPK_U], int b) {
#pragma unroll
      for (int u = 0; u < TOPK_U; ++u) {
        const int vi = b + u * TOPK_NT + lane;
        d[u] = vi < hi ? ldg_na(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint4 q[TOPK_U];
    fetch(q, lo + warp * 32);
    for (int base = lo + warp * 32; base < hi; base += TOPK_U * TOPK_NT) {  // warp-uniform
      uint4 nq[TOPK_U];
      fetch(nq, base + TOPK_U * TOPK_NT);  // the next round, in flight while this one is weighed
#pragma unroll
      for (int u = 0; u < TOPK_U; ++u) {
        const int vi = base + u * TOPK_NT + lane;
        if (vi < hi) {
          const float vm1 = st.m;
          const float vm = online_vec16<DT>(q[u], p.c, st);
          const bool a1 = vm > vm1;
          vm2 = a1 ? vm1 : fmaxf(vm2, vm);
          j1 = a1 ? vi : j1;
        }
      }
#pragma unroll
      for (int u = 0; u < TOPK_U; ++u) q[u] = nq[u];
    }
    m = st.m;
    s = st.sum();
    tmax = st.m;
    // the best vector again (from L2) into the thread's shared slot, an
    // asynchronous copy in flight while the threshold is found
    if (j1 >= 0) cp_async16(&sh.pv[tid], rv + j1);
    cp_async_commit();
  } else {
    for (int i = lo + tid; i < hi; i += TOPK_NT) {
      const float x = Elem<DT>::load(row, i);
      topk_online(x, p.c, m, s);
      tmax = fmaxf(tmax, x);
    }
  }

  // the threshold t: a lower bound of the slice's k-th best element.  The
  // 32 groups of TOPK_GS consecutive threads each have a maximum, an element
  // of the group; k groups have a maximum >= the k-th largest group maximum,
  // so at least k elements are >= it.  Every warp sorts the 32 group maxima
  // itself and takes the k-th: one barrier.
  {
    float g = tmax;
#pragma unroll
    for (int o = 1; o < TOPK_GS; o <<= 1) g = fmaxf(g, __shfl_xor_sync(0xFFFFFFFFu, g, o));
    if (lane % TOPK_GS == 0) sh.gmax[tid / TOPK_GS] = g;
  }
  __syncthreads();
  const float t = __shfl_sync(0xFFFFFFFFu, warp_sort_desc(sh.gmax[lane], lane), k - 1);

  // candidates: the elements >= t.  They lie in the vectors of "hot" threads
  // (their own maximum reaches t).  With vector loads a hot thread whose
  // other vectors all stay below t offers the elements of its best vector
  // (fetched above); one whose other vectors may reach t too (always so
  // when t = -inf) re-reads all its vectors instead: the warp loads such a
  // lane's vectors together, one per lane, HB lanes at a time.  Keys >= t
  // are appended to a shared buffer.
  {
    unsigned hot;
    if (VEC) {
      cp_async_wait_all();  // every thread: no copy outlives this step
      const bool mine = lo + warp * 32 + lane < hi && tmax >= t;
      const bool reread = mine && (j1 < 0 || vm2 >= t);
      if (mine && !reread) {
        float f[VE];
        Elem<DT>::unpack(sh.pv[tid], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          if (f[e] >= t) {
            const int slot = atomicAdd(&sh.nbuf, 1);
            if (slot < TOPK_BUF) sh.buf[slot] = topk_key(f[e], j1 * VE + e);
          }
        }
      }
      hot = __ballot_sync(0xFFFFFFFFu, reread);
    } else {
      hot = __ballot_sync(0xFFFFFFFFu, tmax >= t);
    }
    if (VEC) {
      constexpr int HB = 4;
      const uint4 *rv = reinterpret_cast<const uint4 *>(row);
      const int wfirst = lo + warp * 32;  // lane h's vectors: wfirst + h + j * TOPK_NT
      while (hot) {  // warp-uniform
        int first[HB];
#pragma unroll
        for (int g = 0; g < HB; ++g) {
          first[g] = hot ? wfirst + __ffs(hot) - 1 : hi;  // hi: no lane in this slot
          hot &= hot - 1u;
        }
        // first[0] is the smallest, so its vectors bound the others'
        for (int j0 = 0; first[0] + j0 * TOPK_NT < hi; j0 += 32) {  // warp-uniform
          uint4 q[HB];
          int vi[HB];
#pragma unroll
          for (int g = 0; g < HB; ++g) {
            vi[g] = first[g] + (j0 + lane) * TOPK_NT;
            q[g] = vi[g] < hi ? __ldg(rv + vi[g]) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int g = 0; g < HB; ++g) {
            if (vi[g] >= hi) continue;
            float f[VE];
            Elem<DT>::unpack(q[g], f);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              if (f[e] >= t) {
                const int slot = atomicAdd(&sh.nbuf, 1);
                if (slot < TOPK_BUF) sh.buf[slot] = topk_key(f[e], vi[g] * VE + e);
              }
            }
          }
        }
      }
    }
    while (!VEC && hot) {
      const int h = __ffs(hot) - 1;
      hot &= hot - 1u;
      {
        const int first = lo + warp * 32 + h;  // lane h's elements: first + j * TOPK_NT (see pass 1)
        for (int j0 = 0; first + j0 * TOPK_NT < hi; j0 += 32) {
          const int i = first + (j0 + lane) * TOPK_NT;
          if (i < hi) {
            const float x = Elem<DT>::load(row, i);
            if (x >= t) {
              const int slot = atomicAdd(&sh.nbuf, 1);
              if (slot < TOPK_BUF) sh.buf[slot] = topk_key(x, i);
            }
          }
        }
      }
    }
  }

  // the slice's normalisers: each warp's (their latency overlaps the
  // barrier's wait), then warp 0 combines the warps'
  group_ms(m, s, p.c, 32);
  if (lane == 0) {
    sh.wm[warp] = m;
    sh.ws[warp] = s;
  }
  __syncthreads();

  // the CTA's k best: at most 32 candidates (the usual case) are ranked by
  // warp 0 alone, which stores them straight into rank 0's list; more are
  // ranked by the whole CTA into sh.ctak (or, past the buffer, found by
  // lockstep admission)
  const int nb = sh.nbuf;
  const bool few = nb <= 32;
  if (!few) {
    if (nb <= TOPK_BUF) {
      for (int i = tid; i < nb; i += TOPK_NT) {
        const unsigned long long key = sh.buf[i];
        int rk = 0;
        for (int j = 0; j < nb; ++j) rk += sh.buf[j] > key;
        if (rk < k) sh.ctak[rk] = key;
      }
      __syncthreads();
    } else {
      topk_slice_by_admission<DT, VEC>(row, lo, hi, k, sh);
    }
  }
  if (warp == 0) {
    unsigned long long key;
    int rk;
    if (few) {
      key = lane < nb ? sh.buf[lane] : 0ull;
      rk = lane;  // lanes >= nb: empty slots (key 0) after the nb real keys
      if (lane < nb) {
        rk = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) rk += j < nb && sh.buf[j] > key;
      }
    } else {
      key = lane < k ? sh.ctak[lane] : 0ull;
      rk = lane;
    }
    if (rk < k) dsmem_st_u64(dsmem_addr(&sh.ck[rank][rk], 0), key);
    m = lane < TOPK_NWARP ? sh.wm[lane] : -INFINITY;
    s = lane < TOPK_NWARP ? sh.ws[lane] : 0.f;
    group_ms(m, s, p.c, TOPK_NWARP);
    if (lane == 0) {
      dsmem_st_f32(dsmem_addr(&sh.cm[rank], 0), m);
      dsmem_st_f32(dsmem_addr(&sh.cs[rank], 0), s);
    }
  }
  if (G > 1)
    cluster_sync();  // G is the same for every CTA of the grid
  else
    __syncwarp();  // one CTA per row: warp 0 stored its own list above
  if (tid == 0) topk_stamp(p, 1, false);
  if (rank != 0 || warp != 0) return;
  topk_write_row(p, r, G, k, sh.ck, sh.cm, sh.cs, lane, false);
  __syncwarp();
  if (lane == 0) topk_stamp(p, 2, false);
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
// then rank; parents become list positions.  The parents and values are read
// once into shared memory; depths come from walks there.  Dynamic shared
// memory: key[M] (8 B), parent[M], depth[M], rank[M] (4 B each), byrank[m].
__global__ void __launch_bounds__(NT) rerank_kernel(EagleParams p) {
  extern __shared__ __align__(128) unsigned char rerank_smem[];
  unsigned long long *key = reinterpret_cast<unsigned long long *>(rerank_smem);
  int *spar = reinterpret_cast<int *>(key + p.M);
  int *depth = spar + p.M;
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
    spar[c] = u;
    key[c] = __float_as_uint(__ldg(val + c));  // the value's bits, until the depth is known
    if (c == 0 ? u != -1 : (u < 0 || u >= c)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (!bad) {
    for (int c = tid; c < M; c += NT) {  // parent[c] < c: the walk ends at the root
      int d = 0;
      for (int u = c; u != 0; u = spar[u]) ++d;
      depth[c] = d;
    }
    __syncthreads();
    for (int c = tid; c < M; c += NT)
      key[c] = c == 0 ? 0ull
                      : (static_cast<unsigned long long>(float_order(__uint_as_float(static_cast<uint32_t>(key[c]))))
                         << 32) |
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
      const int u = spar[byrank[r]];
      if (u != 0 && rank[u] >= m) atomicOr(&bad, 1);
    }
    __syncthreads();
  }
  // the kept nodes' tokens, fetched now so that the loads overlap the list
  // positions below (ranks r = tid + i * NT; the rest is read at the end)
  constexpr int TOK_REGS = 4;
  int tkr[TOK_REGS];
#pragma unroll
  for (int i = 0; i < TOK_REGS; ++i) {
    const int r = tid + i * NT;
    tkr[i] = (!bad && r < m) ? __ldg(tok + byrank[r]) : -1;
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
  // (depth, rank); written to key[] of that node for the parent remap.  The
  // depths by rank go to rank[] first (its ranks are no longer needed).
  __syncthreads();
  for (int r = tid; r < m; r += NT) rank[r] = depth[byrank[r]];
  __syncthreads();
  for (int r = tid; r < m; r += NT) {
    const int d = rank[r];
    int q = 1;
    for (int r2 = 0; r2 < m; ++r2) {
      const int d2 = rank[r2];
      q += d2 < d || (d2 == d && r2 < r);
    }
    key[byrank[r]] = static_cast<unsigned long long>(q);  // key[] reused: list position
  }
  __syncthreads();
  if (tid == 0) {
    op[0] = -1;
    ot[0] = __ldg(tok);
    oi[0] = 0;
  }
  for (int r = tid, i = 0; r < m; r += NT, ++i) {
    const int c = byrank[r];
    const int q = static_cast<int>(key[c]);
    const int u = spar[c];
    op[q] = u == 0 ? 0 : static_cast<int>(key[u]);
    int t = -1;
#pragma unroll
    for (int i2 = 0; i2 < TOK_REGS; ++i2)
      if (i2 == i) t = tkr[i2];
    ot[q] = i < TOK_REGS ? t : __ldg(tok + c);
    oi[q] = c;
  }
}

}  // namespace spec
