// n-gram (prompt-lookup) drafting over the context of each sequence
// (glukhov.org, "Спекулятивное декодирование: ускорение инференса LLM на
// 20–50%", §"Спекулятивное декодирование на n-граммах" and §"Настройка
// параметров"; anhtu.dev, "Speculative Decoding: Cách LLM Sinh Văn Bản Nhanh
// Gấp 2–3 Lần", §"Bật trong production").
//
// For sequence b with context t[0 .. len-1], an occurrence of the last n
// tokens ending at e (e <= len - 2, so a token follows it) exists iff
// m(e) >= n, where m(e) is the length of the common suffix of t[.. e] and
// t[.. len-1], clipped to n_max.  With hits(n) = #{e : m(e) >= n}, the draft
// follows latest(n*) = max{e : m(e) >= n*}, n* the largest n in
// [n_min, n_max] with hits(n) >= min_hits.  Equivalently n* is the
// min_hits-th largest value of m over the hits (m >= n_min), so:
//   * min_hits == 1: n* and latest(n*) are the lexicographic maximum of the
//     keys (m(e), e) -- one 64-bit running maximum per thread;
//   * otherwise: a histogram of m (count and latest e per value) decides it,
//     held in registers per thread when n_max - n_min < 8, else in shared
//     memory.
//
// Grid: G CTAs per sequence (G sized from the resident CTAs per SM: 4 for
// the maximum key, at most 64 registers, so that a batch of long contexts
// fits in one wave; 2 for the register histogram; 3 otherwise), each scanning a
// contiguous slice of the end positions with 16-byte loads (U groups of four
// tokens per lane per round, the next round in flight while one is
// compared; the first round is issued before the suffix is in shared
// memory).  t[e] is compared with the last token; only a hit walks back.
// Each CTA reduces its threads' state to a partial.  With G <= 8 the
// sequence's CTAs form one thread-block cluster: the partials go into rank
// 0's shared memory (distributed shared memory stores) and, after one
// cluster barrier, rank 0 combines them and writes the draft.  With larger G
// the partials go to global memory and the last CTA of the sequence to
// finish (a per-sequence counter, put back to zero by that CTA) combines
// them.  One launch.
#pragma once

#include <cstdint>

#include "kernels.cuh"

namespace spec {

constexpr int NGRAM_MAX_N = 64;   // largest n_max
constexpr int NGRAM_U = 4;        // 4-token groups each lane loads per round
constexpr int NGRAM_REG_BINS = 8; // register histogram: n_max - n_min < 8
constexpr int ST_LENGTH = 8;      // device status: lengths[b] outside [0, L]

// per-thread hit bookkeeping
enum NgramMode : int { NGRAM_MAXKEY = 0, NGRAM_REGHIST = 1, NGRAM_SMEMHIST = 2 };

struct NgramParams {
  const int32_t *tokens;   // [B, L]
  const int32_t *lengths;  // [B]
  int B, L, n_min, n_max, min_hits, K;
  int G;                   // CTAs per sequence
  int32_t *out_draft;      // [B, K]
  int32_t *out_count;      // [B]
  int32_t *status;
  void *partials;          // [B, G] partials (u64 key, or 2 * nb ints)
  int *done;               // [B] finished-CTA counters, zero between calls
};

constexpr int NGRAM_MAX_CLUSTER = 8;  // CTAs per sequence that combine through a cluster

struct NgramShared {
  int suf[NGRAM_MAX_N];                 // suf[i] = t[len - 1 - i]
  int cnt[NGRAM_MAX_N + 1];             // histogram: #e with m(e) == k
  int last[NGRAM_MAX_N + 1];            //            latest such e, -1 if none
  unsigned long long wkey[NWARP];
  int is_last;
  int start, count;
  // rank 0 of a cluster: the CTAs' partials (key; or counts and latest e per bin)
  unsigned long long ckey[NGRAM_MAX_CLUSTER];
  int ccnt[NGRAM_MAX_CLUSTER][NGRAM_MAX_N];
  int clast[NGRAM_MAX_CLUSTER][NGRAM_MAX_N];
};

// Four tokens t[4g .. 4g+3]; positions at or past e_end are never compared,
// so what they load does not matter (VEC: rows 16-byte aligned and L % 4 == 0,
// which keeps the whole vector inside the row).
template <bool VEC>
__device__ __forceinline__ int4 ngram_load_group(const int32_t *t, int g, bool live, int e_end) {
  int4 v = make_int4(0, 0, 0, 0);
  if (!live) return v;
  const int e0 = 4 * g;
  if (VEC) {
    v = __ldg(reinterpret_cast<const int4 *>(t) + g);
  } else {
    // live: e0 < e_end, so the clamped indices stay inside the context
    v.x = __ldg(t + e0);
    v.y = __ldg(t + min(e0 + 1, e_end - 1));
    v.z = __ldg(t + min(e0 + 2, e_end - 1));
    v.w = __ldg(t + min(e0 + 3, e_end - 1));
  }
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

template <bool VEC, int MODE, bool CLUSTER>
__global__ void __launch_bounds__(NT, MODE == NGRAM_REGHIST ? 2 : (MODE == NGRAM_MAXKEY ? 4 : 3)) ngram_kernel(NgramParams p) {
  __shared__ NgramShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G;
  const int b = blockIdx.x / G;
  const int rank = blockIdx.x - b * G;
  const int nb = p.n_max - p.n_min + 1;  // histogram bins n_min .. n_max
  pdl_launch_dependents();
  if (MODE == NGRAM_SMEMHIST) {
    for (int k = tid; k <= p.n_max; k += NT) {
      sh.cnt[k] = 0;
      sh.last[k] = -1;
    }
  }
  pdl_wait();
  const int len = __ldg(p.lengths + b);
  const bool bad = len < 0 || len > p.L;
  const int32_t *t = p.tokens + static_cast<size_t>(b) * p.L;
  const int nsuf = bad ? 0 : min(p.n_max, len);
  for (int i = tid; i < nsuf; i += NT) sh.suf[i] = __ldg(t + len - 1 - i);

  const int e_end = bad ? 0 : len - 1;  // end positions e < e_end
  const int ngroups = (max(e_end, 0) + 3) >> 2;
  const int per = (ngroups + G - 1) / G;
  const int g_lo = min(ngroups, rank * per);
  const int g_hi = min(ngroups, g_lo + per);

  unsigned long long key = 0;                  // NGRAM_MAXKEY: max of (m << 32 | e)
  int rc[NGRAM_REG_BINS], rl[NGRAM_REG_BINS];  // NGRAM_REGHIST: count / latest e of m = n_min + k
#pragma unroll
  for (int k = 0; k < NGRAM_REG_BINS; ++k) {
    rc[k] = 0;
    rl[k] = -1;
  }

  // the first round of context loads is in flight while the suffix lands;
  // pv is the group just before the warp's first group of the round (the
  // walk-back window of lane 0)
  int g0 = g_lo + warp * 32 * NGRAM_U;
  int4 v[NGRAM_U];
#pragma unroll
  for (int j = 0; j < NGRAM_U; ++j) {
    const int g = g0 + j * 32 + lane;
    v[j] = ngram_load_group<VEC>(t, g, g < g_hi, e_end);
  }
  int4 pv = ngram_load_group<VEC>(t, g0 - 1, g0 >= 1 && g0 - 1 < g_hi, e_end);
  __syncthreads();
  const int s0 = sh.suf[0];
  int sq[8];  // sq[q] = suf[q]; compared only for q < min(n_max, len)
#pragma unroll
  for (int q = 1; q < 8; ++q) sq[q] = sh.suf[q];
  for (; g0 < g_hi; g0 += NT * NGRAM_U) {  // warp-uniform
    int4 nv[NGRAM_U];                      // next round, loaded before this one is compared
#pragma unroll
    for (int j = 0; j < NGRAM_U; ++j) {
      const int g = g0 + NT * NGRAM_U + j * 32 + lane;
      nv[j] = ngram_load_group<VEC>(t, g, g < g_hi, e_end);
    }
    const int g1 = g0 + NT * NGRAM_U - 1;
    const int4 npv = ngram_load_group<VEC>(t, g1, g1 < g_hi, e_end);
#pragma unroll
    for (int j = 0; j < NGRAM_U; ++j) {
      const int g = g0 + j * 32 + lane;
      // w[0..7] = t[4g-4 .. 4g+3]: the previous group from the lane before
      // (lane 0: the last lane of the previous j, or pv for j == 0)
      int4 prev;
      prev.x = __shfl_up_sync(0xFFFFFFFFu, v[j].x, 1);
      prev.y = __shfl_up_sync(0xFFFFFFFFu, v[j].y, 1);
      prev.z = __shfl_up_sync(0xFFFFFFFFu, v[j].z, 1);
      prev.w = __shfl_up_sync(0xFFFFFFFFu, v[j].w, 1);
      {
        const int4 src = j == 0 ? pv : v[j > 0 ? j - 1 : 0];
        const int4 c31 = make_int4(__shfl_sync(0xFFFFFFFFu, src.x, j == 0 ? 0 : 31),
                                   __shfl_sync(0xFFFFFFFFu, src.y, j == 0 ? 0 : 31),
                                   __shfl_sync(0xFFFFFFFFu, src.z, j == 0 ? 0 : 31),
                                   __shfl_sync(0xFFFFFFFFu, src.w, j == 0 ? 0 : 31));
        if (lane == 0) prev = j == 0 ? pv : c31;
      }
      const int w[8] = {prev.x, prev.y, prev.z, prev.w, v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 4 * g + u;
        if (g < g_hi && e < e_end && w[4 + u] == s0) {
          // matches t[e - q] == suf[q] for q = 1, 2, ...: from the window
          // while it lasts (q <= 4 + u), then from memory
          int mm = 1;
          bool go = true;
#pragma unroll
          for (int q = 1; q < 8; ++q) {
            if (q <= 4 + u) {
              go = go && mm < p.n_max && mm <= e && w[4 + u - q] == sq[q];
              mm += go ? 1 : 0;
            }
          }
          if (go)
            while (mm < p.n_max && mm <= e && __ldg(t + e - mm) == sh.suf[mm]) ++mm;
          if (mm >= p.n_min) {
            if (MODE == NGRAM_MAXKEY) {
              const unsigned long long kk =
                  (static_cast<unsigned long long>(mm) << 32) | static_cast<unsigned>(e);
              key = kk > key ? kk : key;
            } else if (MODE == NGRAM_REGHIST) {
#pragma unroll
              for (int k = 0; k < NGRAM_REG_BINS; ++k)
                if (mm == p.n_min + k) {
                  ++rc[k];
                  rl[k] = max(rl[k], e);
                }
            } else {
              atomicAdd(&sh.cnt[mm], 1);
              atomicMax(&sh.last[mm], e);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NGRAM_U; ++j) v[j] = nv[j];
    pv = npv;
  }

  // this CTA's partial
  if (MODE == NGRAM_MAXKEY) {
    key = warp_max_u64(key);
    if (lane == 0) sh.wkey[warp] = key;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0;
      for (int w = 0; w < NWARP; ++w) m = sh.wkey[w] > m ? sh.wkey[w] : m;
      if (CLUSTER)
        dsmem_st_u64(dsmem_addr(&sh.ckey[rank], 0), m);
      else
        static_cast<unsigned long long *>(p.partials)[blockIdx.x] = m;
    }
  } else {
    if (MODE == NGRAM_REGHIST) {
      if (tid <= p.n_max) {
        sh.cnt[tid] = 0;
        sh.last[tid] = -1;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < NGRAM_REG_BINS; ++k) {
        if (k < nb) {  // uniform
          const int c = __reduce_add_sync(0xFFFFFFFFu, rc[k]);
          const int l = __reduce_max_sync(0xFFFFFFFFu, rl[k]);
          if (lane == 0 && c > 0) {
            atomicAdd(&sh.cnt[p.n_min + k], c);
            atomicMax(&sh.last[p.n_min + k], l);
          }
        }
      }
    }
    __syncthreads();
    if (CLUSTER) {
      for (int k = tid; k < nb; k += NT) {
        dsmem_st_s32(dsmem_addr(&sh.ccnt[rank][k], 0), sh.cnt[p.n_min + k]);
        dsmem_st_s32(dsmem_addr(&sh.clast[rank][k], 0), sh.last[p.n_min + k]);
      }
    } else {
      int *part = static_cast<int *>(p.partials) + static_cast<size_t>(blockIdx.x) * 2 * nb;
      for (int k = tid; k < nb; k += NT) {
        part[k] = sh.cnt[p.n_min + k];
        part[nb + k] = sh.last[p.n_min + k];
      }
    }
  }
  if (CLUSTER) {
    // rank 0 of the cluster combines the G partials in its shared memory
    cluster_sync();
    if (rank != 0) return;
  } else {
    // the last CTA of the sequence to finish combines the partials
    __threadfence();
    __syncthreads();
    if (tid == 0) sh.is_last = atomicAdd(p.done + b, 1) == G - 1;
    __syncthreads();
    if (!sh.is_last) return;
    __threadfence();
    if (tid == 0) p.done[b] = 0;  // ready for the next call on this workspace
  }

  int start = -1;
  if (MODE == NGRAM_MAXKEY) {
    const unsigned long long *parts =
        static_cast<const unsigned long long *>(p.partials) + static_cast<size_t>(b) * G;
    unsigned long long m = 0;
    for (int r = tid; r < G; r += NT) {
      const unsigned long long x = CLUSTER ? sh.ckey[r] : __ldcg(parts + r);
      m = x > m ? x : m;
    }
    m = warp_max_u64(m);
    if (lane == 0) sh.wkey[warp] = m;
    __syncthreads();
    if (tid == 0) {
      for (int w = 0; w < NWARP; ++w) m = sh.wkey[w] > m ? sh.wkey[w] : m;
      if (m != 0) start = static_cast<int>(m & 0xFFFFFFFFu) + 1;
    }
  } else {
    if (CLUSTER) {
      // bin by bin over the G CTAs: the sequence's totals into sh.cnt / sh.last
      for (int k = tid; k < nb; k += NT) {
        int c = 0, l = -1;
        for (int r = 0; r < G; ++r) {
          c += sh.ccnt[r][k];
          l = max(l, sh.clast[r][k]);
        }
        sh.cnt[p.n_min + k] = c;
        sh.last[p.n_min + k] = l;
      }
    } else {
      for (int k = tid; k <= p.n_max; k += NT) {
        sh.cnt[k] = 0;
        sh.last[k] = -1;
      }
      __syncthreads();
      const int *parts = static_cast<const int *>(p.partials) + static_cast<size_t>(b) * G * 2 * nb;
      for (int i = tid; i < G * nb; i += NT) {
        const int r = i / nb, k = i - r * nb;
        const int c = __ldcg(parts + static_cast<size_t>(r) * 2 * nb + k);
        if (c > 0) {
          atomicAdd(&sh.cnt[p.n_min + k], c);
          atomicMax(&sh.last[p.n_min + k], __ldcg(parts + static_cast<size_t>(r) * 2 * nb + nb + k));
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      int hits = 0, latest = -1;
      for (int n = p.n_max; n >= p.n_min; --n) {
        hits += sh.cnt[n];
        latest = max(latest, sh.last[n]);
        if (hits >= p.min_hits) {
          start = latest + 1;
          break;
        }
      }
    }
  }
  if (tid == 0) {
    int count = 0;
    if (bad) {
      count = -1;
      atomicOr(p.status, ST_LENGTH);
    } else if (start >= 0) {
      count = min(len - start, p.K);
    }
    sh.start = start;
    sh.count = count;
    p.out_count[b] = count;
  }
  __syncthreads();
  int32_t *d = p.out_draft + static_cast<size_t>(b) * p.K;
  for (int k = tid; k < p.K; k += NT) d[k] = k < sh.count ? __ldg(t + sh.start + k) : -1;
}

}  // namespace spec
