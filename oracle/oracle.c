/*
 * Reference oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  The product path
 * (the CUDA library under sampling_row_online_gb300/) never calls it, and
 * the two share no code: no headers, no helpers, no constants.
 *
 * Everything here is deliberately plain: fp64 arithmetic, left-to-right
 * loops, no blocking, no fusion, no reordering.  Each function names the
 * passage of the source pages it restates.  The pages cited are
 *   [Oscine]  blog.oscine.io, "投机解码：让大模型「猜」着跑的数学魔术"
 *   [Anhtu]   anhtu.dev, "Speculative Decoding: Cách LLM Sinh Văn Bản
 *             Nhanh Gấp 2–3 Lần"
 *   [Infra53] infra-guide, "5.3 Medusa, EAGLE và MTP"
 *   [Glukhov] glukhov.org, "Спекулятивное декодирование: ускорение
 *             инференса LLM на 20–50%"
 * The random numbers follow Salmon, Moraes, Dror and Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3" (SC'11), Philox4x32 with 10 rounds.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes of the repository):
 *   - temperature T enters as p = softmax(z_t / T), q = softmax(z_d / T),
 *     the same T for both; T == 0 selects greedy matching.
 *   - "accept with probability min(1, p/q)" is taken as: accept iff u < p/q,
 *     u uniform on the 2^-24 grid [0, 1 - 2^-24].
 *   - q(x) == 0: accept iff p(x) > 0 (ratio +inf); 0/0 counts as a reject.
 *   - residual mass Z == 0 after a reject: sample from p at that position
 *     with the same uniform (counted as a fallback).
 *   - inverse-CDF: the smallest v with C(v) > t, C the running sum in index
 *     order; if none (rounding), the largest v with positive weight.
 *   - argmax ties go to the lowest index.
 *   - uniform for (seed, b, position, slot): Philox4x32-10 with key
 *     (seed mod 2^32, seed >> 32), counter (b, position, slot, 0), and
 *     u = (word0 >> 8) * 2^-24.  Slot 0 = acceptance, slot 1 = residual
 *     or bonus sample.  The bonus uses position K.
 *
 * Parity pins: every public function here is pinned by a CPU test against
 * something other than itself (known-answer vectors, closed forms, exact
 * enumeration, chi-square, hand cases, brute force); see tests/.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* status codes (values chosen to match nothing in particular) */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_TOKEN 2
#define ORC_ERR_PARENT 3

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11, section 4.2 / Figure 2).        */
/* One round: two 32x32->64 products of the even words with the round  */
/* multipliers; the odd words are xored with the high halves and the   */
/* round key; the key advances by the Weyl constants between rounds.   */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mul0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)mul1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* u = (x >> 8) * 2^-24 on word 0 of Philox(counter=(b,position,slot,0),
 * key=(seed lo, seed hi)). */
double oracle_uniform(uint64_t seed, uint32_t b, uint32_t position,
                      uint32_t slot) {
  uint32_t ctr[4] = {b, position, slot, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------ */
/* logits: dtype 0 = IEEE fp32, 1 = bfloat16 (upper half of an fp32).   */
/* Both widen to double exactly.                                        */
/* ------------------------------------------------------------------ */
static double logit_at(const void *z, int dtype, int64_t i) {
  float f;
  if (dtype == 0) {
    f = ((const float *)z)[i];
  } else {
    uint32_t bits = (uint32_t)((const uint16_t *)z)[i] << 16;
    memcpy(&f, &bits, sizeof f);
  }
  return (double)f;
}

static const void *row_ptr(const void *base, int dtype, int64_t row,
                           int64_t V) {
  size_t esz = dtype == 0 ? 4u : 2u;
  return (const char *)base + (size_t)row * (size_t)V * esz;
}

/* Row normalisers of p = softmax(z / T) ([Oscine] §"验收标准的精确数学":
 * p is the target's next-token distribution, q the draft's):
 *   m = max_v z[v],  S = sum_v exp((z[v] - m) / T), summed left to right. */
void oracle_row_stats(const void *z, int dtype, int V, double T, double *m_out,
                      double *S_out) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(z, dtype, v);
    if (x > m) m = x;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) S += exp((logit_at(z, dtype, v) - m) / T);
  *m_out = m;
  *S_out = S;
}

/* p(v) for one row given its normalisers. */
static double prob_at(const void *z, int dtype, int v, double T, double m,
                      double S) {
  return exp((logit_at(z, dtype, v) - m) / T) / S;
}

/* First index of the maximum ([Infra53] §9.1 names greedy matching as its
 * own acceptance rule: the draft must equal the target's top token). */
int oracle_argmax(const void *z, int dtype, int V) {
  int best = 0;
  double bv = logit_at(z, dtype, 0);
  for (int v = 1; v < V; ++v) {
    double x = logit_at(z, dtype, v);
    if (x > bv) {
      bv = x;
      best = v;
    }
  }
  return best;
}

/* Acceptance test ([Oscine] §"验收标准的精确数学", eq. α(x) and its two
 * cases; [Anhtu] §"Toán học của sự miễn phí", first bullet):
 * accept x with probability min(1, p(x)/q(x)), realised as u < p/q.
 * Returns 1 for accept; *r_out gets p/q (may be +inf); *near_out is set
 * when |u - r| <= 1e-5 * max(r, 2^-24). */
int oracle_accept(const void *zt, const void *zd, int dtype, int V, double T,
                  int x, double u, double *r_out, int *near_out) {
  double mt, St, md, Sd;
  oracle_row_stats(zt, dtype, V, T, &mt, &St);
  oracle_row_stats(zd, dtype, V, T, &md, &Sd);
  double p = prob_at(zt, dtype, x, T, mt, St);
  double q = prob_at(zd, dtype, x, T, md, Sd);
  double r;
  if (q > 0.0)
    r = p / q;
  else
    r = p > 0.0 ? INFINITY : 0.0;
  if (r_out) *r_out = r;
  if (near_out) {
    double scale = r > 0x1p-24 ? r : 0x1p-24;
    *near_out = isfinite(r) && fabs(u - r) <= 1e-5 * scale;
  }
  return u < r;
}

/* Inverse-CDF draw over non-negative weights w[0..V-1] with total Z:
 * t = u * Z; the smallest v with C(v) > t, where C is the running sum in
 * index order; if none, the largest v with w[v] > 0.  *near_out is set
 * when t lies within 1e-5 * Z of C(v*) or of C(v*-1) (C(-1) = 0). */
static int inverse_cdf(const double *w, int V, double Z, double u,
                       int *near_out) {
  double t = u * Z;
  double C = 0.0, Cprev = 0.0;
  int pick = -1;
  for (int v = 0; v < V; ++v) {
    Cprev = C;
    C += w[v];
    if (C > t) {
      pick = v;
      break;
    }
  }
  if (pick < 0) {
    for (int v = V - 1; v >= 0; --v)
      if (w[v] > 0.0) {
        pick = v;
        break;
      }
    if (pick < 0) pick = 0;
    Cprev = C;
  }
  if (near_out)
    *near_out = fabs(t - C) <= 1e-5 * Z || fabs(t - Cprev) <= 1e-5 * Z;
  return pick;
}

/* Sample from p itself (the bonus token of [Anhtu] §"Toán học của sự miễn
 * phí", third bullet, and [Oscine] §"多 Token 验证", step 4): weights
 * exp((z - m)/T) with Z = S. */
int oracle_target_sample(const void *zt, int dtype, int V, double T, double u,
                         int *near_out) {
  double m, S;
  oracle_row_stats(zt, dtype, V, T, &m, &S);
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  for (int v = 0; v < V; ++v) w[v] = exp((logit_at(zt, dtype, v) - m) / T);
  int tok = inverse_cdf(w, V, S, u, near_out);
  free(w);
  return tok;
}

/* Residual resample after a reject ([Oscine] §"拒绝之后怎么办？——残差分布",
 * eq. p_resid; [Glukhov] §"Математическая гарантия", eq. r(x)):
 * w(v) = max(0, p(v) - q(v)), Z = sum_v w(v), draw from w / Z.
 * If Z == 0 the draw falls back to p at this position (*fallback_out = 1). */
int oracle_residual_sample(const void *zt, const void *zd, int dtype, int V,
                           double T, double u, int *near_out,
                           int *fallback_out) {
  double mt, St, md, Sd;
  oracle_row_stats(zt, dtype, V, T, &mt, &St);
  oracle_row_stats(zd, dtype, V, T, &md, &Sd);
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  double Z = 0.0;
  for (int v = 0; v < V; ++v) {
    double d = prob_at(zt, dtype, v, T, mt, St) - prob_at(zd, dtype, v, T, md, Sd);
    w[v] = d > 0.0 ? d : 0.0;
    Z += w[v];
  }
  int tok;
  if (Z > 0.0) {
    tok = inverse_cdf(w, V, Z, u, near_out);
    if (fallback_out) *fallback_out = 0;
  } else {
    tok = oracle_target_sample(zt, dtype, V, T, u, near_out);
    if (fallback_out) *fallback_out = 1;
  }
  free(w);
  return tok;
}

/* ------------------------------------------------------------------ */
/* One sequence of the chain verification ([Oscine] §"多 Token 验证：左到  */
/* 右，遇错即停"; [Anhtu] §"Toán học của sự miễn phí"):                    */
/*   for i = 0..K-1: accept x_i with min(1, p_i/q_i); on the first reject */
/*   resample from the residual at i and stop;                          */
/*   if all K are accepted, draw the bonus from p_K.                    */
/* T == 0 is greedy matching ([Infra53] §9.1): x_i is kept iff it equals */
/* argmax p_i; the first mismatch emits argmax p_i; a full match emits   */
/* argmax p_K.                                                           */
/* Output: tokens[0..n-1] = x, tokens[n] = the new token, rest -1;       */
/* returns n (number of accepted drafts) or -1 on a token out of range.  */
/* u_acc[i] / u_samp[j] override the Philox uniforms when non-NULL.      */
/* ------------------------------------------------------------------ */
static int verify_one(const void *zt_seq, const void *zd_seq,
                      const int32_t *x, int K, int V, int dtype, double T,
                      uint64_t seed, uint32_t b, const double *u_acc,
                      const double *u_samp, int32_t *tokens, int *near_out,
                      int *fallback_out) {
  int near = 0, fallback = 0;
  for (int i = 0; i <= K; ++i) tokens[i] = -1;
  for (int i = 0; i < K; ++i)
    if (x[i] < 0 || x[i] >= V) {
      if (near_out) *near_out = 0;
      if (fallback_out) *fallback_out = 0;
      return -1;
    }
  int n = K, tok = -1;
  for (int i = 0; i < K; ++i) {
    const void *zt = row_ptr(zt_seq, dtype, i, V);
    if (T == 0.0) {
      int a = oracle_argmax(zt, dtype, V);
      if (x[i] != a) {
        n = i;
        tok = a;
        break;
      }
      continue;
    }
    const void *zd = row_ptr(zd_seq, dtype, i, V);
    double u = u_acc ? u_acc[i] : oracle_uniform(seed, b, (uint32_t)i, 0u);
    int nr = 0;
    int ok = oracle_accept(zt, zd, dtype, V, T, x[i], u, NULL, &nr);
    near |= nr;
    if (!ok) {
      double us = u_samp ? u_samp[i] : oracle_uniform(seed, b, (uint32_t)i, 1u);
      int ns = 0, fb = 0;
      tok = oracle_residual_sample(zt, zd, dtype, V, T, us, &ns, &fb);
      near |= ns;
      fallback |= fb;
      n = i;
      break;
    }
  }
  if (n == K) {
    const void *zt = row_ptr(zt_seq, dtype, K, V);
    if (T == 0.0) {
      tok = oracle_argmax(zt, dtype, V);
    } else {
      double us = u_samp ? u_samp[K] : oracle_uniform(seed, b, (uint32_t)K, 1u);
      int ns = 0;
      tok = oracle_target_sample(zt, dtype, V, T, us, &ns);
      near |= ns;
    }
  }
  for (int i = 0; i < n; ++i) tokens[i] = x[i];
  tokens[n] = tok;
  if (near_out) *near_out = near;
  if (fallback_out) *fallback_out = fallback;
  return n;
}

/* Batched chain verification over nb sequences.
 *   zt: [nb, K+1, V], zd: [nb, K, V] (ignored when T == 0), x: [nb, K]
 *   b_ids: the sequence index b that keys the uniforms of each of the nb
 *          sequences (NULL: b = 0..nb-1)
 *   u_acc: [nb, K], u_samp: [nb, K+1] optional injected uniforms
 *   out_tokens: [nb, K+1], out_n: [nb], out_near/out_fallback: [nb] or NULL
 *   out_m, out_S: [nb, 2K+1] or NULL; row order = target rows 0..K, then
 *          draft rows 0..K-1 (S is not computed when T == 0).
 * Returns ORC_OK, or ORC_ERR_TOKEN when any sequence had a token outside
 * [0, V) (its out_n is -1 and its tokens are -1). */
int oracle_verify_chain(const void *zt, const void *zd, const int32_t *x,
                        int nb, int K, int V, int dtype, double T,
                        uint64_t seed, const int32_t *b_ids,
                        const double *u_acc, const double *u_samp,
                        int32_t *out_tokens, int32_t *out_n, int32_t *out_near,
                        int32_t *out_fallback, double *out_m, double *out_S,
                        int nthreads) {
  if (nb < 0 || K < 0 || V <= 0 || (dtype != 0 && dtype != 1) || !(T >= 0.0))
    return ORC_ERR_ARG;
  int status = ORC_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) \
    reduction(max : status)
  for (int s = 0; s < nb; ++s) {
    uint32_t b = b_ids ? (uint32_t)b_ids[s] : (uint32_t)s;
    const void *zt_seq = row_ptr(zt, dtype, (int64_t)s * (K + 1), V);
    const void *zd_seq = zd ? row_ptr(zd, dtype, (int64_t)s * K, V) : NULL;
    int near = 0, fb = 0;
    int n = verify_one(zt_seq, zd_seq, x + (size_t)s * K, K, V, dtype, T, seed,
                       b, u_acc ? u_acc + (size_t)s * K : NULL,
                       u_samp ? u_samp + (size_t)s * (K + 1) : NULL,
                       out_tokens + (size_t)s * (K + 1), &near, &fb);
    out_n[s] = n;
    if (n < 0) status = ORC_ERR_TOKEN;
    if (out_near) out_near[s] = near;
    if (out_fallback) out_fallback[s] = fb;
    if (out_m || out_S) {
      int R = 2 * K + 1;
      for (int r = 0; r < R; ++r) {
        /* draft rows are not part of greedy matching: NaN when T == 0 */
        const void *row = r <= K ? row_ptr(zt_seq, dtype, r, V)
                                 : (zd_seq && T > 0.0 ? row_ptr(zd_seq, dtype, r - K - 1, V)
                                                      : NULL);
        double m = NAN, S = NAN;
        if (row) {
          if (T > 0.0) {
            oracle_row_stats(row, dtype, V, T, &m, &S);
          } else {
            m = logit_at(row, dtype, oracle_argmax(row, dtype, V));
          }
        }
        if (out_m) out_m[(size_t)s * R + r] = m;
        if (out_S) out_S[(size_t)s * R + r] = S;
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Verification of drafts from a deterministic drafter: the n-gram        */
/* drafter ([Glukhov] §"Спекулятивное декодирование на n-граммах")       */
/* proposes tokens, not a distribution.  Reading taken: the chain rule    */
/* ([Oscine] §"验收标准的精确数学", §"拒绝之后怎么办？——残差分布") with    */
/* q_i the point mass at x_i: accept x_i iff u < p_i(x_i); at the first   */
/* reject j draw from max(0, p_j - q_j), i.e. p_j with x_j removed        */
/* (weights exp((z_j(v) - m_j)/T) for v != x_j); if all k drafts of the   */
/* sequence are accepted, the bonus comes from p_k.  Each sequence has    */
/* its own draft count k = counts[s] in [0, K] (NULL: K); drafts past it  */
/* are not read.  Uniforms as the chain: (b, i, 0) for the test of x_i,   */
/* (b, n, 1) for the draw at n.  T == 0: greedy matching of the k drafts. */
/*   zt: [nb, K+1, V], x: [nb, K], out_tokens: [nb, K+1], out_n: [nb]     */
/* ------------------------------------------------------------------ */
int oracle_verify_points(const void *zt, const int32_t *x, const int32_t *counts,
                         int nb, int K, int V, int dtype, double T, uint64_t seed,
                         const int32_t *b_ids, int32_t *out_tokens, int32_t *out_n,
                         int32_t *out_near, int nthreads) {
  if (nb < 0 || K < 0 || V <= 0 || (dtype != 0 && dtype != 1) || !(T >= 0.0))
    return ORC_ERR_ARG;
  int status = ORC_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) \
    reduction(max : status)
  for (int s = 0; s < nb; ++s) {
    uint32_t b = b_ids ? (uint32_t)b_ids[s] : (uint32_t)s;
    const void *zt_seq = row_ptr(zt, dtype, (int64_t)s * (K + 1), V);
    const int32_t *xs = x + (size_t)s * K;
    int32_t *tokens = out_tokens + (size_t)s * (K + 1);
    int k = counts ? counts[s] : K;
    int near = 0, bad = k < 0 || k > K;
    for (int i = 0; i <= K; ++i) tokens[i] = -1;
    for (int i = 0; !bad && i < k; ++i)
      if (xs[i] < 0 || xs[i] >= V) bad = 1;
    if (bad) {
      out_n[s] = -1;
      if (out_near) out_near[s] = 0;
      status = ORC_ERR_TOKEN;
      continue;
    }
    int n = k, tok = -1;
    double *w = T > 0.0 ? (double *)malloc(sizeof(double) * (size_t)V) : NULL;
    for (int i = 0; i < k; ++i) {
      const void *row = row_ptr(zt_seq, dtype, i, V);
      if (T == 0.0) {
        int a = oracle_argmax(row, dtype, V);
        if (xs[i] != a) {
          n = i;
          tok = a;
          break;
        }
        continue;
      }
      double m, S;
      oracle_row_stats(row, dtype, V, T, &m, &S);
      double r = prob_at(row, dtype, xs[i], T, m, S); /* p(x) / q(x), q(x) = 1 */
      double u = oracle_uniform(seed, b, (uint32_t)i, 0u);
      double scale = r > 1.0 / 16777216.0 ? r : 1.0 / 16777216.0;
      if (fabs(u - r) <= 1e-5 * scale) near = 1;
      if (!(u < r)) {
        double Z = 0.0;
        for (int v = 0; v < V; ++v) {
          w[v] = v == xs[i] ? 0.0 : exp((logit_at(row, dtype, v) - m) / T);
          Z += w[v];
        }
        int nr = 0;
        tok = inverse_cdf(w, V, Z, oracle_uniform(seed, b, (uint32_t)i, 1u), &nr);
        near |= nr;
        n = i;
        break;
      }
    }
    if (n == k) {
      const void *row = row_ptr(zt_seq, dtype, k, V);
      if (T == 0.0) {
        tok = oracle_argmax(row, dtype, V);
      } else {
        int nr = 0;
        tok = oracle_target_sample(row, dtype, V, T, oracle_uniform(seed, b, (uint32_t)k, 1u), &nr);
        near |= nr;
      }
    }
    free(w);
    for (int i = 0; i < n; ++i) tokens[i] = xs[i];
    tokens[n] = tok;
    out_n[s] = n;
    if (out_near) out_near[s] = near;
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Draft tree ([Infra53] §3 and §8: node 0 is the root, every parent     */
/* precedes its child, parent[0] = -1; depth = parent's depth + 1).      */
/* ------------------------------------------------------------------ */
static int check_parent(const int32_t *parent, int N) {
  if (N <= 0 || parent[0] != -1) return 0;
  for (int c = 1; c < N; ++c)
    if (parent[c] < 0 || parent[c] >= c) return 0;
  return 1;
}

/* Largest node depth, or -1 if parent[] is not a valid tree. */
int oracle_tree_max_depth(const int32_t *parent, int N) {
  if (!check_parent(parent, N)) return -1;
  int *depth = (int *)malloc(sizeof(int) * (size_t)N);
  int D = 0;
  depth[0] = 0;
  for (int c = 1; c < N; ++c) {
    depth[c] = depth[parent[c]] + 1;
    if (depth[c] > D) D = depth[c];
  }
  free(depth);
  return D;
}

/* Tree-attention mask and position IDs ([Infra53] §3.1–§3.2 and the
 * worked example of §8): node n sees exactly its ancestors and itself,
 * found by walking parent pointers up to the root; its position ID is its
 * depth.  mask: [N, N] bytes, depth: [N]. */
int oracle_tree_mask(const int32_t *parent, int N, uint8_t *mask,
                     int32_t *depth) {
  if (!check_parent(parent, N)) return ORC_ERR_PARENT;
  memset(mask, 0, (size_t)N * (size_t)N);
  for (int n = 0; n < N; ++n) {
    depth[n] = parent[n] == -1 ? 0 : depth[parent[n]] + 1;
    for (int a = n; a != -1; a = parent[a]) mask[(size_t)n * N + a] = 1;
  }
  return ORC_OK;
}

/* Greedy tree verification ([Anhtu] §"Token tree": the deepest accepted
 * branch is the output; [Infra53] §3.2: only one path is committed;
 * [Infra53] §9.1: greedy matching).  Row n of zt is the target's
 * distribution after node n, so node c (c >= 1) is accepted iff its parent
 * is accepted and node_tokens[c] == argmax(row parent[c]).  The committed
 * path ends at the deepest accepted node (lowest index among equals); the
 * output is the path's tokens (root excluded) followed by the bonus
 * argmax(row d*), padded with -1 to max_depth + 1 entries.
 *   zt: [nb, N, V], node_tokens: [nb, N] (entry 0 ignored),
 *   out_path: [nb, max_depth + 1], out_len: [nb] */
int oracle_verify_tree_greedy(const void *zt, const int32_t *parent,
                              const int32_t *node_tokens, int nb, int N, int V,
                              int dtype, int max_depth, int32_t *out_path,
                              int32_t *out_len, int nthreads) {
  if (nb < 0 || N <= 0 || V <= 0 || (dtype != 0 && dtype != 1))
    return ORC_ERR_ARG;
  int D = oracle_tree_max_depth(parent, N);
  if (D < 0) return ORC_ERR_PARENT;
  if (max_depth < D) return ORC_ERR_ARG;
  int W = max_depth + 1;
  int status = ORC_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) \
    reduction(max : status)
  for (int s = 0; s < nb; ++s) {
    const void *zt_seq = row_ptr(zt, dtype, (int64_t)s * N, V);
    const int32_t *tok = node_tokens + (size_t)s * N;
    int32_t *path = out_path + (size_t)s * W;
    for (int k = 0; k < W; ++k) path[k] = -1;
    int bad = 0;
    for (int c = 1; c < N; ++c)
      if (tok[c] < 0 || tok[c] >= V) bad = 1;
    if (bad) {
      out_len[s] = -1;
      status = ORC_ERR_TOKEN;
      continue;
    }
    int *amax = (int *)malloc(sizeof(int) * (size_t)N);
    int *depth = (int *)malloc(sizeof(int) * (size_t)N);
    char *acc = (char *)malloc((size_t)N);
    for (int n = 0; n < N; ++n)
      amax[n] = oracle_argmax(row_ptr(zt_seq, dtype, n, V), dtype, V);
    acc[0] = 1;
    depth[0] = 0;
    int best = 0;
    for (int c = 1; c < N; ++c) {
      int p = parent[c];
      depth[c] = depth[p] + 1;
      acc[c] = acc[p] && tok[c] == amax[p];
      if (acc[c] && depth[c] > depth[best]) best = c;
    }
    int d = depth[best];
    for (int n = best, k = d - 1; n != 0; n = parent[n], --k) path[k] = tok[n];
    path[d] = amax[best];
    out_len[s] = d + 1;
    free(amax);
    free(depth);
    free(acc);
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Stochastic tree verification.  The pages give the chain rule          */
/* ([Oscine] §"验收标准的精确数学" and §"拒绝之后怎么办？——残差分布") and    */
/* warn that verifying a tree does not by itself keep the output          */
/* lossless ([Infra53] §9); the rule for several children of one node is  */
/* not given.  Reading taken, the lossless extension of the chain rule:   */
/* the children of a node are candidates drawn independently from the     */
/* draft's distribution q at that node and are tried in index order.      */
/* With r the current target distribution at the node (r = p at first), */
/* candidate x is accepted with probability min(1, r(x)/q(x)); on a       */
/* reject r becomes norm(max(0, r - q)) and the next candidate is tried.  */
/* An accepted candidate becomes the current node; a node whose           */
/* candidates are all rejected emits a draw from r; an accepted node with */
/* no children emits a bonus draw from its own p.                         */
/* After k rejects at a node r = max(0, p - a_k q) / W_k with a_0 = 0,     */
/* W_0 = 1, a_{k+1} = a_k + W_k and W_{k+1} = sum_v max(0, p - a_{k+1} q) */
/* (max(0, r - q) = max(0, p - (a_k + W_k) q) / W_k).                     */
/* Uniforms: the test of child c uses (b, c - 1, slot 0), the draw at     */
/* node u uses (b, u, slot 1); on a chain-shaped tree (parent[c] = c - 1) */
/* this is exactly the chain verification of the same rows.               */
/* A residual that vanishes after a reject (W == 0, through rounding      */
/* only) ends the node: the draw falls back to p there (*fallback).       */
/*   zt, zd: [nb, N, V] (row u: target / draft distribution at node u;    */
/*   leaves' draft rows are not read), node_tokens: [nb, N] (entry 0      */
/*   ignored), u_acc / u_samp: [nb, N] optional injected uniforms (test   */
/*   of child c, draw at node u), out_path: [nb, max_depth + 1] (accepted */
/*   tokens, then the emitted token, -1 padding), out_len: [nb] (accepted */
/*   + 1, or -1 on a token outside [0, V)).                               */
/* ------------------------------------------------------------------ */
static int verify_tree_one(const void *zt_seq, const void *zd_seq,
                           const int32_t *parent, const int32_t *tok, int N,
                           int V, int dtype, double T, uint64_t seed,
                           uint32_t b, const double *u_acc,
                           const double *u_samp, int32_t *path, int W,
                           int *near_out, int *fallback_out) {
  int near = 0, fallback = 0, len = 0;
  for (int k = 0; k < W; ++k) path[k] = -1;
  for (int c = 1; c < N; ++c)
    if (tok[c] < 0 || tok[c] >= V) {
      *near_out = 0;
      *fallback_out = 0;
      return -1;
    }
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  int u = 0, emitted = -1;
  for (;;) {
    const void *zt = row_ptr(zt_seq, dtype, u, V);
    double mt, St;
    oracle_row_stats(zt, dtype, V, T, &mt, &St);
    int first = -1;
    for (int c = u + 1; c < N; ++c)
      if (parent[c] == u) {
        first = c;
        break;
      }
    double us = u_samp ? u_samp[u] : oracle_uniform(seed, b, (uint32_t)u, 1u);
    if (first < 0) {  /* a leaf: the bonus token from p */
      int ns = 0;
      emitted = oracle_target_sample(zt, dtype, V, T, us, &ns);
      near |= ns;
      break;
    }
    const void *zd = row_ptr(zd_seq, dtype, u, V);
    double md, Sd;
    oracle_row_stats(zd, dtype, V, T, &md, &Sd);
    double a = 0.0, Wk = 1.0;
    int next = -1, vanished = 0;
    for (int c = first; c < N; ++c) {
      if (parent[c] != u) continue;
      int x = tok[c];
      double px = prob_at(zt, dtype, x, T, mt, St);
      double qx = prob_at(zd, dtype, x, T, md, Sd);
      double rx = px - a * qx;
      if (rx < 0.0) rx = 0.0;
      rx /= Wk;
      double ratio;
      if (qx > 0.0)
        ratio = rx / qx;
      else
        ratio = rx > 0.0 ? INFINITY : 0.0;
      double uc = u_acc ? u_acc[c] : oracle_uniform(seed, b, (uint32_t)(c - 1), 0u);
      double scale = ratio > 0x1p-24 ? ratio : 0x1p-24;
      if (isfinite(ratio) && fabs(uc - ratio) <= 1e-5 * scale) near = 1;
      if (uc < ratio) {
        next = c;
        break;
      }
      /* reject: r <- norm(max(0, r - q)) */
      a += Wk;
      double Z = 0.0;
      for (int v = 0; v < V; ++v) {
        double d = prob_at(zt, dtype, v, T, mt, St) - a * prob_at(zd, dtype, v, T, md, Sd);
        w[v] = d > 0.0 ? d : 0.0;
        Z += w[v];
      }
      Wk = Z;
      if (!(Wk > 0.0)) {
        vanished = 1;
        break;
      }
    }
    if (next >= 0) {
      path[len++] = tok[next];
      u = next;
      continue;
    }
    int ns = 0;
    if (vanished || a == 0.0) {  /* a == 0 cannot happen: u has a child */
      emitted = oracle_target_sample(zt, dtype, V, T, us, &ns);
      fallback |= vanished;
    } else {
      emitted = inverse_cdf(w, V, Wk, us, &ns);
    }
    near |= ns;
    break;
  }
  free(w);
  path[len] = emitted;
  *near_out = near;
  *fallback_out = fallback;
  return len + 1;
}

int oracle_verify_tree_sample(const void *zt, const void *zd,
                              const int32_t *parent, const int32_t *node_tokens,
                              int nb, int N, int V, int dtype, double T,
                              uint64_t seed, int max_depth,
                              const int32_t *b_ids, const double *u_acc,
                              const double *u_samp, int32_t *out_path,
                              int32_t *out_len, int32_t *out_near,
                              int32_t *out_fallback, int nthreads) {
  if (nb < 0 || N <= 0 || V <= 0 || (dtype != 0 && dtype != 1) || !(T > 0.0))
    return ORC_ERR_ARG;
  int D = oracle_tree_max_depth(parent, N);
  if (D < 0) return ORC_ERR_PARENT;
  if (max_depth < D) return ORC_ERR_ARG;
  int W = max_depth + 1;
  int status = ORC_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) \
    reduction(max : status)
  for (int s = 0; s < nb; ++s) {
    uint32_t b = b_ids ? (uint32_t)b_ids[s] : (uint32_t)s;
    int near = 0, fb = 0;
    int len = verify_tree_one(row_ptr(zt, dtype, (int64_t)s * N, V),
                              row_ptr(zd, dtype, (int64_t)s * N, V), parent,
                              node_tokens + (size_t)s * N, N, V, dtype, T,
                              seed, b, u_acc ? u_acc + (size_t)s * N : NULL,
                              u_samp ? u_samp + (size_t)s * N : NULL,
                              out_path + (size_t)s * W, W, &near, &fb);
    out_len[s] = len;
    if (len < 0) status = ORC_ERR_TOKEN;
    if (out_near) out_near[s] = near;
    if (out_fallback) out_fallback[s] = fb;
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* n-gram (prompt-lookup) drafter ([Glukhov] §"Спекулятивное             */
/* декодирование на n-граммах": find an earlier occurrence of the current */
/* n-gram in the context and propose the tokens that followed it;        */
/* [Anhtu] §"Bật trong production": prompt_lookup_max bounds the n-gram   */
/* window, num_speculative_tokens is K; [Glukhov] §"Настройка            */
/* параметров" and the llama.cpp flags beside it: min-hits, the number of */
/* times the pattern must have been seen).  Reading taken: the longest n  */
/* in [n_min, n_max] whose last-n-token suffix occurred at least min_hits */
/* times earlier wins, and of its occurrences the most recent one (the    */
/* largest start j with j + n <= len - 1, so at least one token follows   */
/* it); the proposal is the up to K tokens after that occurrence.         */
/* Written as the plain search: n from n_max down, every start j from the */
/* end down, token by token.                                              */
/*   tokens: [B, L] int32 (row b holds lengths[b] <= L tokens),           */
/*   out_draft: [B, K] (proposal, -1 padding), out_count: [B].            */
/* ------------------------------------------------------------------ */
int oracle_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B,
                         int L, int n_min, int n_max, int min_hits, int K,
                         int32_t *out_draft, int32_t *out_count) {
  if (B < 0 || L < 0 || n_min < 1 || n_max < n_min || min_hits < 1 || K < 0) return ORC_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const int32_t *t = tokens + (size_t)b * L;
    int len = lengths[b];
    if (len < 0 || len > L) return ORC_ERR_ARG;
    int32_t *d = out_draft + (size_t)b * K;
    for (int k = 0; k < K; ++k) d[k] = -1;
    int start = -1;
    for (int n = n_max; n >= n_min && start < 0; --n) {
      if (n > len - 1) continue;
      int hits = 0, recent = -1;
      for (int j = len - n - 1; j >= 0; --j) {
        int same = 1;
        for (int i = 0; i < n; ++i)
          if (t[j + i] != t[len - n + i]) {
            same = 0;
            break;
          }
        if (same) {
          if (recent < 0) recent = j;
          ++hits;
        }
      }
      if (hits >= min_hits) start = recent + n;
    }
    int count = 0;
    if (start >= 0) {
      count = len - start < K ? len - start : K;
      for (int k = 0; k < count; ++k) d[k] = t[start + k];
    }
    out_count[b] = count;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* EAGLE-2 tree budget ([Infra53] §5.1-§5.3: the draft's confidence     */
/* decides where a limited node budget goes; a node's value is the       */
/* product of the confidences on its path from the root; an expansion    */
/* phase grows the few best nodes, a rerank phase keeps the best nodes   */
/* of all for verification).  Readings taken: a confidence is the        */
/* draft's probability of the token, softmax(z / T) of the draft row at  */
/* the parent; every frontier node offers its k most probable tokens as  */
/* candidates; the k_next candidates of highest value become the next    */
/* frontier; the rerank keeps the root and the m highest-valued nodes of  */
/* all candidates.                                                        */
/* ------------------------------------------------------------------ */

/* Top-k of each of R rows by logit (ties: lower index first), with each
 * token's probability under softmax(z / T).  Plain selection: k passes,
 * each taking the largest logit not taken yet. */
int oracle_topk_prob(const void *z, int R, int V, int dtype, double T, int k,
                     int32_t *out_tok, double *out_prob) {
  if (R < 0 || V < 1 || k < 1 || k > V || !(T > 0.0)) return ORC_ERR_ARG;
  unsigned char *taken = (unsigned char *)malloc((size_t)V);
  if (!taken) return ORC_ERR_ARG;
  for (int r = 0; r < R; ++r) {
    const void *row = row_ptr(z, dtype, r, V);
    double m, S;
    oracle_row_stats(row, dtype, V, T, &m, &S);
    memset(taken, 0, (size_t)V);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      double bv = 0.0;
      for (int v = 0; v < V; ++v) {
        if (taken[v]) continue;
        double x = logit_at(row, dtype, v);
        if (best < 0 || x > bv) {
          best = v;
          bv = x;
        }
      }
      taken[best] = 1;
      out_tok[(size_t)r * k + j] = best;
      out_prob[(size_t)r * k + j] = prob_at(row, dtype, best, T, m, S);
    }
  }
  free(taken);
  return ORC_OK;
}

/* Does candidate a rank above candidate b: higher value, ties to the
 * lower index. */
static int ranks_above(double va, int ia, double vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

static int near_gap(double a, double b) {
  double hi = fabs(a) > fabs(b) ? fabs(a) : fabs(b);
  return fabs(a - b) <= 1e-5 * hi;
}

/* One expansion step for B trees.  Node arrays per tree ([B, cap]):
 * node_tok, node_val, node_par.  frontier [B, F] holds node ids; the
 * candidates of frontier node f are written to nodes offset + f*k + j
 * (j = 0..k-1, the row's top-k in order) with value
 * node_val[frontier] * prob and parent frontier.  out_next [B, k_next]
 * receives the k_next new candidates of highest value (ties: lower node
 * id), best first.  out_near[b] flags a selection boundary where the
 * k_next-th and the next value lie within 1e-5 (relative). */
int oracle_eagle2_expand(const int32_t *frontier, int B, int F, int k,
                         const int32_t *topk_tok, const double *topk_prob,
                         int32_t *node_tok, double *node_val, int32_t *node_par,
                         int cap, int offset, int k_next, int32_t *out_next,
                         uint8_t *out_near) {
  if (B < 0 || F < 1 || k < 1 || offset < 1 || offset + F * k > cap ||
      k_next < 0 || k_next > F * k)
    return ORC_ERR_ARG;
  int n = F * k;
  unsigned char *taken = (unsigned char *)malloc((size_t)n);
  if (!taken) return ORC_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    int32_t *tok = node_tok + (size_t)b * cap;
    double *val = node_val + (size_t)b * cap;
    int32_t *par = node_par + (size_t)b * cap;
    for (int f = 0; f < F; ++f) {
      int u = frontier[(size_t)b * F + f];
      if (u < 0 || u >= offset) {
        free(taken);
        return ORC_ERR_ARG;
      }
      for (int j = 0; j < k; ++j) {
        int c = offset + f * k + j;
        tok[c] = topk_tok[((size_t)b * F + f) * k + j];
        val[c] = val[u] * topk_prob[((size_t)b * F + f) * k + j];
        par[c] = u;
      }
    }
    memset(taken, 0, (size_t)n);
    double last = 0.0;
    for (int s = 0; s < k_next; ++s) {
      int best = -1;
      for (int i = 0; i < n; ++i)
        if (!taken[i] && (best < 0 || ranks_above(val[offset + i], i, val[offset + best], best)))
          best = i;
      taken[best] = 1;
      out_next[(size_t)b * k_next + s] = offset + best;
      last = val[offset + best];
    }
    out_near[b] = 0;
    if (k_next > 0 && k_next < n) {
      for (int i = 0; i < n; ++i)
        if (!taken[i] && near_gap(val[offset + i], last)) out_near[b] = 1;
    }
  }
  free(taken);
  return ORC_OK;
}

/* Rerank for B trees of M nodes (node 0 the root, parent[c] < c): keep
 * the root and the m other nodes of highest value, ties to the smaller
 * depth, then the lower node id.  A child's value never exceeds its
 * parent's (a probability is at most 1), so the kept set holds every
 * ancestor of a kept node.  The kept nodes are listed by depth, then in
 * rank order; out_par holds parents as positions in that list (-1 for the
 * root), out_tok their tokens, out_idx their node ids.  out_near[b] flags
 * a boundary where the m-th kept value and a dropped one lie within 1e-5.
 * Returns ORC_ERR_PARENT if a tree is malformed or a kept node's parent
 * was dropped (values that grow along a path). */
int oracle_eagle2_rerank(const double *node_val, const int32_t *node_par,
                         const int32_t *node_tok, int B, int M, int m,
                         int32_t *out_par, int32_t *out_tok, int32_t *out_idx,
                         uint8_t *out_near) {
  if (B < 0 || M < 1 || m < 0 || m > M - 1) return ORC_ERR_ARG;
  int *depth = (int *)malloc(sizeof(int) * (size_t)M);
  int *rank_of = (int *)malloc(sizeof(int) * (size_t)M);
  int *order = (int *)malloc(sizeof(int) * (size_t)M);
  int *pos = (int *)malloc(sizeof(int) * (size_t)M);
  if (!depth || !rank_of || !order || !pos) {
    free(depth); free(rank_of); free(order); free(pos);
    return ORC_ERR_ARG;
  }
  int status = ORC_OK;
  for (int b = 0; b < B && status == ORC_OK; ++b) {
    const double *val = node_val + (size_t)b * M;
    const int32_t *par = node_par + (size_t)b * M;
    const int32_t *tok = node_tok + (size_t)b * M;
    if (par[0] != -1) { status = ORC_ERR_PARENT; break; }
    depth[0] = 0;
    for (int c = 1; c < M; ++c) {
      if (par[c] < 0 || par[c] >= c) { status = ORC_ERR_PARENT; break; }
      depth[c] = depth[par[c]] + 1;
    }
    if (status != ORC_OK) break;
    /* selection: rank r = the r-th best non-root node */
    for (int c = 0; c < M; ++c) rank_of[c] = -1;
    double last = 0.0;
    for (int r = 0; r < m; ++r) {
      int best = -1;
      for (int c = 1; c < M; ++c) {
        if (rank_of[c] >= 0) continue;
        if (best < 0 || val[c] > val[best] ||
            (val[c] == val[best] && (depth[c] < depth[best] ||
                                     (depth[c] == depth[best] && c < best))))
          best = c;
      }
      rank_of[best] = r;
      last = val[best];
    }
    out_near[b] = 0;
    if (m > 0)
      for (int c = 1; c < M; ++c)
        if (rank_of[c] < 0 && near_gap(val[c], last)) out_near[b] = 1;
    /* listing: root, then by depth, then by rank */
    int n = 0;
    order[n++] = 0;
    int maxd = 0;
    for (int c = 1; c < M; ++c) if (depth[c] > maxd) maxd = depth[c];
    for (int d = 1; d <= maxd; ++d)
      for (int r = 0; r < m; ++r)
        for (int c = 1; c < M; ++c)
          if (rank_of[c] == r && depth[c] == d) order[n++] = c;
    for (int c = 0; c < M; ++c) pos[c] = -1;
    for (int i = 0; i < n; ++i) pos[order[i]] = i;
    int32_t *op = out_par + (size_t)b * (m + 1);
    int32_t *ot = out_tok + (size_t)b * (m + 1);
    int32_t *oi = out_idx + (size_t)b * (m + 1);
    for (int i = 0; i < n; ++i) {
      int c = order[i];
      oi[i] = c;
      ot[i] = tok[c];
      if (c == 0) {
        op[i] = -1;
      } else {
        op[i] = pos[par[c]];
        if (op[i] < 0) status = ORC_ERR_PARENT;
      }
    }
  }
  free(depth); free(rank_of); free(order); free(pos);
  return status;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
