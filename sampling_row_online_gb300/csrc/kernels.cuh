// Verification kernels for sm_103a.
//
// One thread-block cluster per "job", one job per logit row (or row pair):
//   chain, T > 0 : job i < K reads target row i and draft row i together,
//                  job K reads the bonus target row K;
//   chain, T = 0 : job i reads target row i (argmax only);
//   tree         : job n reads target row n (argmax only).
// The C CTAs of a cluster split the vocabulary into C slices; each CTA
// streams its slice from HBM into shared memory with TMA bulk copies
// (cp.async.bulk + mbarrier), reduces it, and the cluster combines the
// partial results through distributed shared memory.  Everything a job
// needs after the row statistics (the acceptance test, the residual or bonus
// draw) runs on the data still held on chip, so each logit is read from HBM
// once.  The last job of a sequence to finish (an atomic ticket) writes the
// sequence's outputs.
//
// Method (pages cited by title and section):
//   blog.oscine.io "投机解码：让大模型「猜」着跑的数学魔术":
//     §"验收标准的精确数学" (accept with min(1, p/q)),
//     §"拒绝之后怎么办？——残差分布" (residual norm(max(0, p - q))),
//     §"多 Token 验证：左到右，遇错即停" (left-to-right stop, bonus token);
//   anhtu.dev "Speculative Decoding: Cách LLM Sinh Văn Bản Nhanh Gấp 2–3 Lần",
//     §"Toán học của sự miễn phí" and §"Token tree";
//   infra-guide "5.3 Medusa, EAGLE và MTP", §3 (tree, one committed path)
//     and §9.1 (greedy matching).
#pragma once

#include <cfloat>
#include <cstdint>

#include "philox.cuh"
#include "ptx.cuh"

namespace spec {

constexpr int NT = 256;                 // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int VECS_PER_THREAD = 2;      // 16-byte vectors per thread per tile
constexpr int MAX_STAGES = 8;
constexpr int MAX_TILES = 64;
constexpr int MAX_CLUSTER = 16;
constexpr int FIRST_REJ_NONE = 0x7F7F7F7F;  // also the byte pattern the workspace is memset to
constexpr int CAND_FALLBACK = 1 << 30;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s bound on any wait

// device status bits (per stream)
constexpr int ST_TOKEN = 1, ST_PARENT = 2, ST_TIMEOUT = 4;

enum Kind : int { KIND_SAMPLE = 0, KIND_GREEDY_CHAIN = 1, KIND_TREE = 2 };

struct Stats {  // layout-compatible with spec_stats_t
  unsigned long long sequences, accepted, bonus, resampled, residual_fallbacks, errors;
};

struct Params {
  const void *zt;           // [B, J, V] target rows (J = K+1 chain, N tree)
  const void *zd;           // [B, K, V] draft rows (sampling only)
  const int32_t *tokens;    // chain: draft tokens [B, K]; tree: node tokens [B, N]
  const int32_t *parent;    // tree: [N]
  int B, K, V, J;           // K = drafts (chain) or N (tree)
  int kind;
  float c;                  // log2(e) / T
  uint64_t seed;
  int slice;                // vocabulary elements per CTA (multiple of the vector width)
  int tile;                 // elements per tile and row
  int stages;               // shared-memory stages of the tile ring
  int ncl;                  // clusters launched (persistent)
  int njobs;                // jobs in total
  int emit_off;             // byte offset of the emission scratch in dynamic smem
  int max_depth;            // tree output width - 1
  int32_t *out_tokens;      // chain [B, K+1]; tree [B, max_depth+1]
  int32_t *out_n;           // chain n_accepted [B]; tree length [B]
  float *out_row_max;       // [B, 2K+1] or null
  float *out_row_sumexp;    // [B, 2K+1] or null
  Stats *stats;             // or null
  int32_t *ticket;          // [B] jobs finished (reset by the last one)
  int32_t *first_rej;       // [B] lowest rejected position (reset by the last job)
  int32_t *seq_err;         // [B] error flags (reset by the last job)
  int32_t *cand;            // [B, J] per-job result token
  int32_t *status;          // device status bits
};

// ------------------------------------------------------------------ elements
template <int DT>
struct Elem;

template <>
struct Elem<0> {  // fp32
  static constexpr int VE = 4;
  static constexpr int BYTES = 4;
  __device__ static __forceinline__ void unpack(const uint4 v, float (&f)[VE]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ float load(const unsigned char *row, int i) {
    return __ldg(reinterpret_cast<const float *>(row) + i);
  }
  __device__ static __forceinline__ void store_neg_inf(unsigned char *p) {
    *reinterpret_cast<uint32_t *>(p) = 0xFF800000u;
  }
  __device__ static __forceinline__ void copy_elem(unsigned char *dst, const unsigned char *src) {
    *reinterpret_cast<uint32_t *>(dst) = __ldg(reinterpret_cast<const unsigned int *>(src));
  }
};

template <>
struct Elem<1> {  // bfloat16: the upper half of an fp32
  static constexpr int VE = 8;
  static constexpr int BYTES = 2;
  __device__ static __forceinline__ void unpack(const uint4 v, float (&f)[VE]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
  __device__ static __forceinline__ float load(const unsigned char *row, int i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(row) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ static __forceinline__ void store_neg_inf(unsigned char *p) {
    *reinterpret_cast<uint16_t *>(p) = 0xFF80u;
  }
  __device__ static __forceinline__ void copy_elem(unsigned char *dst, const unsigned char *src) {
    *reinterpret_cast<uint16_t *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
  }
};

// ------------------------------------------------------------- reductions
// (max, sum of 2^((z - max) c)) pairs; an empty side has max = -inf, sum = 0.
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float c) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    m = M;
    s = 0.f;
    return;
  }
  s = s * ex2((m - M) * c) + s2 * ex2((m2 - M) * c);
  m = M;
}

// Block-wide (max, sumexp) reduction; the result is valid in thread 0.
// Fixed combination order, so the result is deterministic.
__device__ __forceinline__ void block_reduce_ms(float &m, float &s, float c, float *sh_m,
                                                float *sh_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_down_sync(0xFFFFFFFFu, m, off);
    const float s2 = __shfl_down_sync(0xFFFFFFFFu, s, off);
    ms_combine(m, s, m2, s2, c);
  }
  if (lane == 0) {
    sh_m[warp] = m;
    sh_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    m = sh_m[0];
    s = sh_s[0];
    for (int w = 1; w < NWARP; ++w) ms_combine(m, s, sh_m[w], sh_s[w], c);
  }
  __syncthreads();
}

__device__ __forceinline__ float block_reduce_sum(float v, float *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, off);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float r = 0.f;
  if (threadIdx.x == 0) {
    r = sh[0];
    for (int w = 1; w < NWARP; ++w) r += sh[w];
  }
  __syncthreads();
  return r;
}

// (value, index) maximum with ties to the lower index; index INT_MAX = none.
__device__ __forceinline__ void am_combine(float &v, int &i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void block_reduce_argmax(float &v, int &i, float *shv, int *shi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_down_sync(0xFFFFFFFFu, v, off);
    const int i2 = __shfl_down_sync(0xFFFFFFFFu, i, off);
    am_combine(v, i, v2, i2);
  }
  if (lane == 0) {
    shv[warp] = v;
    shi[warp] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    v = shv[0];
    i = shi[0];
    for (int w = 1; w < NWARP; ++w) am_combine(v, i, shv[w], shi[w]);
  }
  __syncthreads();
}

__device__ __forceinline__ int block_reduce_min_int(int v, int *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_down_sync(0xFFFFFFFFu, v, off));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  int r = sh[0];
  for (int w = 1; w < NWARP; ++w) r = min(r, sh[w]);
  __syncthreads();
  return r;  // valid in every thread
}

__device__ __forceinline__ int block_reduce_max_int(int v, int *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_down_sync(0xFFFFFFFFu, v, off));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  int r = sh[0];
  for (int w = 1; w < NWARP; ++w) r = max(r, sh[w]);
  __syncthreads();
  return r;
}

// Exclusive prefix sum over the threads of the block, in thread order; the
// block total is returned in *total (every thread).  sh: NWARP + 1 floats.
__device__ __forceinline__ float block_exclusive_scan(float v, float *sh, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float n = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc = __fadd_rn(inc, n);
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  float base = 0.f;
  for (int w = 0; w < warp; ++w) base = __fadd_rn(base, sh[w]);
  const float excl = __fadd_rn(base, __fsub_rn(inc, v));
  if (threadIdx.x == NT - 1) sh[NWARP] = __fadd_rn(excl, v);
  __syncthreads();
  *total = sh[NWARP];
  __syncthreads();
  return excl;
}

// -------------------------------------------------------- job stream
// The kernels are persistent: cluster `cl` handles jobs q = cl, cl + ncl,
// cl + 2 ncl, ...  Every CTA of the cluster streams the tiles of its
// vocabulary slice of those jobs, in order, through a ring of S shared-memory
// stages, so the copies of the next job are in flight while the current job
// is combined and decided.  TMA path: thread 0 issues one bulk copy per row
// and tile, one mbarrier per stage tracks completion.  Plain path (rows not
// 16-byte aligned): all threads copy element by element and pad the last
// vector with -inf.

// Job q -> (sequence b, row i).  Stochastic chain: the K row pairs in
// position-major order (so earlier positions of a sequence tend to be decided
// first), then the K+1-th target rows.  Argmax kinds: rows position-major.
__device__ __forceinline__ void decode_job(const Params &p, int q, int &b, int &i) {
  if (p.kind == KIND_SAMPLE) {
    const int npair = p.B * p.K;
    if (q < npair) {
      i = q / p.B;
      b = q - i * p.B;
    } else {
      i = p.K;
      b = q - npair;
    }
  } else {
    i = q / p.B;
    b = q - i * p.B;
  }
}

template <int DT, bool TMA>
struct Stream {
  using E = Elem<DT>;
  const Params *p;
  unsigned char *buf;
  uint64_t *full;
  int cl, lo, len, nt, S, srows;
  bool timed_out;

  __device__ __forceinline__ int tile_len(int k) const { return min(p->tile, len - k * p->tile); }
  __device__ __forceinline__ unsigned char *stage_row(int s, int r) const {
    return buf + static_cast<size_t>(s * srows + r) * p->tile * E::BYTES;
  }
  // target and (for a pair) draft row of job q; returns the row count
  __device__ __forceinline__ int rows_of(int q, const unsigned char *&rt,
                                         const unsigned char *&rd) const {
    int b, i;
    decode_job(*p, q, b, i);
    rt = static_cast<const unsigned char *>(p->zt) +
         (static_cast<size_t>(b) * p->J + i) * p->V * E::BYTES;
    if (p->kind == KIND_SAMPLE && i < p->K) {
      rd = static_cast<const unsigned char *>(p->zd) +
           (static_cast<size_t>(b) * p->K + i) * p->V * E::BYTES;
      return 2;
    }
    rd = nullptr;
    return 1;
  }

  // TMA, thread 0: issue tile `seq` of this CTA's stream, if it exists.
  __device__ __forceinline__ void produce(int seq) {
    if (nt == 0) return;
    const int n = seq / nt, k = seq - n * nt;
    const int q = cl + n * p->ncl;
    if (q >= p->njobs) return;
    const unsigned char *rt, *rd;
    const int nr = rows_of(q, rt, rd);
    const int s = seq % S;
    const uint32_t bytes = static_cast<uint32_t>(tile_len(k)) * E::BYTES;
    const size_t off = (static_cast<size_t>(lo) + static_cast<size_t>(k) * p->tile) * E::BYTES;
    mbar_arrive_expect_tx(&full[s], bytes * nr);
    bulk_g2s(stage_row(s, 0), rt + off, bytes, &full[s]);
    if (nr == 2) bulk_g2s(stage_row(s, 1), rd + off, bytes, &full[s]);
  }

  __device__ __forceinline__ void prologue() {
    if (TMA && threadIdx.x == 0)
      for (int s = 0; s < S; ++s) produce(s);
  }

  // Every thread: tile `seq` (tile k of the current job, rows rt/rd) is in
  // stage seq % S on return.
  __device__ __forceinline__ void acquire(int seq, int k, const unsigned char *rt,
                                          const unsigned char *rd) {
    const int s = seq % S;
    if (TMA) {
      const uint32_t par = static_cast<uint32_t>(seq / S) & 1u;
      if (!mbar_try_wait(&full[s], par)) {
        const uint64_t t0 = clock_ns();
        while (!mbar_try_wait(&full[s], par)) {
          if (clock_ns() - t0 > WAIT_LIMIT_NS) {
            timed_out = true;
            break;
          }
        }
      }
    } else {
      __syncthreads();
      const int n = tile_len(k);
      const int npad = (n + E::VE - 1) / E::VE * E::VE;
      const size_t off = (static_cast<size_t>(lo) + static_cast<size_t>(k) * p->tile) * E::BYTES;
      for (int r = 0; r < (rd ? 2 : 1); ++r) {
        const unsigned char *g = (r ? rd : rt) + off;
        unsigned char *d = stage_row(s, r);
        for (int e = threadIdx.x; e < npad; e += NT) {
          if (e < n)
            E::copy_elem(d + e * E::BYTES, g + e * E::BYTES);
          else
            E::store_neg_inf(d + e * E::BYTES);
        }
      }
      __syncthreads();
    }
  }

  // After every thread consumed tile `seq`: refill its stage with tile seq + S.
  __device__ __forceinline__ void release(int seq) {
    if (TMA) {
      __syncthreads();
      if (threadIdx.x == 0) produce(seq + S);
    }
  }

  // Bounded drain of copies that may still be in flight after a timeout.
  __device__ __forceinline__ void drain_after_timeout(int seq_end) {
    if (!TMA) return;
    const uint64_t t0 = clock_ns();
    for (int seq = seq_end; seq < seq_end + S; ++seq)
      while (!mbar_try_wait(&full[seq % S], static_cast<uint32_t>(seq / S) & 1u) &&
             clock_ns() - t0 < WAIT_LIMIT_NS) {
      }
  }
};

// Online (max, sum 2^((z - max) c)) over one vector of logits.
template <int VE>
__device__ __forceinline__ void online_update(const float (&f)[VE], float c, float &m, float &s,
                                              float &mc) {
  float vm = f[0];
#pragma unroll
  for (int k = 1; k < VE; ++k) vm = fmaxf(vm, f[k]);
  if (vm > m) {
    s *= ex2((m - vm) * c);
    m = vm;
    mc = m * c;
  }
  if (m > -INFINITY) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < VE; ++k) a += ex2(fmaf(f[k], c, -mc));
    s += a;
  }
}

// Weight of one vocabulary entry in the second pass: the residual
// max(0, p - q) of a rejected pair, or the unnormalised p of a draw from p.
// Explicit roundings, so the summation and the search compute identical bits.
struct Weights {
  float c, mtc, mdc, inv_st, inv_sd;
  bool resid;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float et = ex2(fmaf(zt, c, -mtc));
    if (!resid) return et;
    const float ed = ex2(fmaf(zd, c, -mdc));
    return fmaxf(__fsub_rn(__fmul_rn(et, inv_st), __fmul_rn(ed, inv_sd)), 0.f);
  }
};

// --------------------------------------------------------- shared state
struct SharedSmall {
  uint64_t full[MAX_STAGES];
  float red_m[2][NWARP];
  float red_s[2][NWARP];
  // Pushed by every CTA of the cluster into every CTA's copy (st.shared::cluster
  // before the cluster barrier), double-buffered by job parity, so combines
  // read local shared memory only:
  alignas(16) float xs[2][MAX_CLUSTER][4];  // per rank: (m_t, s_t, m_d, s_d) or (max, index bits)
  float xz[2][2][MAX_CLUSTER];              // per rank: slice mass of the draw (round 0 / 1)
  int xhint[2];                             // rank 0: lowest rejected position seen
  // per-job values of this CTA
  float gz[2][2];     // z_t[x], z_d[x]
  int gok[2];         // draft token in range
  float bf[8];        // broadcast floats
  int bi[8];          // broadcast ints
  int scratch[NWARP];
  float fscratch[NWARP + 1];
};

// Ticket of sequence b: true in every thread of the CTA that finished the
// sequence's last job.  Call from every thread of one CTA.
__device__ __forceinline__ bool take_ticket(const Params &p, int b, SharedSmall &sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&p.ticket[b], 1);
    sh.bi[7] = (old == p.J - 1);
    if (old == p.J - 1) __threadfence();
  }
  __syncthreads();
  return sh.bi[7] != 0;
}

// Outputs of stochastic-chain sequence b, once all its jobs are done.
__device__ __forceinline__ void emit_chain_sample(const Params &p, int b) {
  const int err = __ldcg(p.seq_err + b);
  const int n = min(__ldcg(p.first_rej + b), p.K);
  const int cn = __ldcg(p.cand + static_cast<size_t>(b) * p.J + n);
  for (int e = threadIdx.x; e <= p.K; e += NT) {
    int v = -1;
    if (!err) {
      if (e < n)
        v = __ldg(p.tokens + static_cast<size_t>(b) * p.K + e);
      else if (e == n)
        v = cn & ~CAND_FALLBACK;
    }
    p.out_tokens[static_cast<size_t>(b) * (p.K + 1) + e] = v;
  }
  if (threadIdx.x == 0) {
    p.out_n[b] = err ? -1 : n;
    if (p.stats) {
      if (err) {
        atomicAdd(&p.stats->errors, 1ull);
      } else {
        atomicAdd(&p.stats->sequences, 1ull);
        atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(n));
        atomicAdd(n == p.K ? &p.stats->bonus : &p.stats->resampled, 1ull);
        if (n < p.K && (cn & CAND_FALLBACK)) atomicAdd(&p.stats->residual_fallbacks, 1ull);
      }
    }
    p.ticket[b] = 0;
    p.first_rej[b] = FIRST_REJ_NONE;
    p.seq_err[b] = 0;
  }
}

// ======================================================================
// Stochastic chain: row statistics, acceptance test, residual/bonus draw.
// ======================================================================
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT, 3) sample_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ SharedSmall sh;

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const float c = p.c;

  Stream<DT, TMA> st;
  st.p = &p;
  st.buf = dyn;
  st.full = sh.full;
  st.cl = blockIdx.x / C;
  st.lo = static_cast<int>(rank) * p.slice;
  st.len = max(0, min(p.V, st.lo + p.slice) - st.lo);
  st.nt = (st.len + p.tile - 1) / p.tile;
  st.S = p.stages;
  st.srows = p.K > 0 ? 2 : 1;
  st.timed_out = false;
  const int lo = st.lo, len = st.len;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  st.prologue();

  // contiguous chunk of this thread in the second pass
  const int E2 = ((len + NT - 1) / NT + VE - 1) / VE * VE;
  const int e0 = min(len, tid * E2), e1 = min(len, e0 + E2);

  // draft token of the next job, loaded one job ahead by thread 32
  auto token_of = [&](int q) -> int {
    if (q >= p.njobs) return 0;
    int b, i;
    decode_job(p, q, b, i);
    return i < p.K ? __ldg(p.tokens + static_cast<size_t>(b) * p.K + i) : 0;
  };
  int x_next = (tid == 32) ? token_of(st.cl) : 0;

  int seq = 0;
  for (int n = 0;; ++n) {
    const int q = st.cl + n * p.ncl;
    if (q >= p.njobs) break;
    const int par = n & 1;
    int b, i;
    decode_job(p, q, b, i);
    const bool pair = i < p.K;
    const unsigned char *rt, *rd;
    st.rows_of(q, rt, rd);

    // draft token's two logits and the rejection hint: loads issued now by
    // thread 32, consumed after pass 1
    int g_ok = 1, g_hint = 0;
    float g_zt = 0.f, g_zd = 0.f;
    if (tid == 32) {
      const int x = x_next;
      if (pair) {
        g_ok = (x >= 0 && x < p.V);
        if (g_ok) {
          g_zt = E::load(rt, x);
          g_zd = E::load(rd, x);
        }
      }
      if (rank == 0) g_hint = *reinterpret_cast<volatile int *>(p.first_rej + b);
      x_next = token_of(q + p.ncl);
    }

    // ---- pass 1: online max / sum-exp of both rows of this slice
    float mt = -INFINITY, s_t = 0.f, mtc = 0.f;
    float md = -INFINITY, s_d = 0.f, mdc = 0.f;
    for (int k = 0; k < st.nt; ++k, ++seq) {
      st.acquire(seq, k, rt, rd);
      const int s = seq % st.S;
      const int nv = (st.tile_len(k) + VE - 1) / VE;
      const unsigned char *bt = st.stage_row(s, 0);
      if (pair) {
        const unsigned char *bd = st.stage_row(s, 1);
        for (int j = tid; j < nv; j += NT) {
          float f[VE];
          E::unpack(lds128(bt + j * 16), f);
          online_update<VE>(f, c, mt, s_t, mtc);
          E::unpack(lds128(bd + j * 16), f);
          online_update<VE>(f, c, md, s_d, mdc);
        }
      } else {
        for (int j = tid; j < nv; j += NT) {
          float f[VE];
          E::unpack(lds128(bt + j * 16), f);
          online_update<VE>(f, c, mt, s_t, mtc);
        }
      }
      st.release(seq);
    }
    block_reduce_ms(mt, s_t, c, sh.red_m[0], sh.red_s[0]);
    if (pair) block_reduce_ms(md, s_d, c, sh.red_m[1], sh.red_s[1]);
    if (tid < 32) {  // push this slice's statistics into every CTA of the cluster
      const float a0 = __shfl_sync(0xFFFFFFFFu, mt, 0), a1 = __shfl_sync(0xFFFFFFFFu, s_t, 0);
      const float a2 = __shfl_sync(0xFFFFFFFFu, md, 0), a3 = __shfl_sync(0xFFFFFFFFu, s_d, 0);
      if (tid < static_cast<int>(C)) dsmem_st_v4f32(dsmem_addr(&sh.xs[par][rank][0], tid), a0, a1, a2, a3);
    } else if (tid == 32) {
      sh.gok[par] = g_ok;
      sh.gz[par][0] = g_zt;
      sh.gz[par][1] = g_zd;
      if (rank == 0)
        for (uint32_t r = 0; r < C; ++r) dsmem_st_s32(dsmem_addr(&sh.xhint[par], r), g_hint);
    }
    cluster_sync();  // partial statistics of job n visible cluster-wide

    // ---- combine the slices (rank order) and take the acceptance decision
    if (tid == 0) {
      float Mt = -INFINITY, St = 0.f, Md = -INFINITY, Sd = 0.f;
      for (uint32_t r = 0; r < C; ++r) {
        ms_combine(Mt, St, sh.xs[par][r][0], sh.xs[par][r][1], c);
        if (pair) ms_combine(Md, Sd, sh.xs[par][r][2], sh.xs[par][r][3], c);
      }
      const int hint = sh.xhint[par];
      const int ok = sh.gok[par];
      int accept = 1;
      if (pair && ok) {
        const float a = fmaf(sh.gz[par][0], c, -(Mt * c));
        const float d = fmaf(sh.gz[par][1], c, -(Md * c));
        const float ratio = ex2(a - d) * (Sd / St);  // p_i(x_i) / q_i(x_i)
        const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u);
        accept = u < ratio;
      }
      const int need = pair ? (ok && !accept) : 1;
      const int superseded = pair ? (hint < i) : (hint < p.K);
      sh.bi[0] = need && !superseded;
      sh.bf[0] = Mt;
      sh.bf[1] = St;
      sh.bf[2] = Md;
      sh.bf[3] = Sd;
      if (rank == 0) {
        const int R = 2 * p.K + 1;
        if (p.out_row_max) {
          p.out_row_max[static_cast<size_t>(b) * R + i] = Mt;
          if (pair) p.out_row_max[static_cast<size_t>(b) * R + p.K + 1 + i] = Md;
        }
        if (p.out_row_sumexp) {
          p.out_row_sumexp[static_cast<size_t>(b) * R + i] = St;
          if (pair) p.out_row_sumexp[static_cast<size_t>(b) * R + p.K + 1 + i] = Sd;
        }
        if (pair && !ok) {
          atomicOr(p.seq_err + b, 1);
          atomicOr(p.status, ST_TOKEN);
        }
        if (pair && ok && !accept) atomicMin(p.first_rej + b, i);
      }
    }
    __syncthreads();

    int taker = 0;  // the CTA that records the job and takes its ticket
    if (sh.bi[0]) {
      // ---- pass 2 (a reject or the bonus row), from the slice just read
      // (L2-resident): per-thread contiguous chunks, block scan, slice mass,
      // cluster exchange, owner slice, then one thread walks its chunk.
      Weights W;
      W.c = c;
      W.mtc = sh.bf[0] * c;
      W.mdc = sh.bf[2] * c;
      W.inv_st = 1.f / sh.bf[1];
      W.inv_sd = 1.f / sh.bf[3];
      W.resid = pair;
      int fallback = 0, owner = 0, pl = 0;
      float tl = 0.f, excl = 0.f, sum = 0.f;
      for (int round = 0; round < 2; ++round) {
        sum = 0.f;
        if (TMA) {
#pragma unroll 4
          for (int e = e0; e < e1; e += VE) {
            const size_t off = static_cast<size_t>(lo + e) * E::BYTES;
            float ft[VE], fd[VE];
            E::unpack(__ldg(reinterpret_cast<const uint4 *>(rt + off)), ft);
            if (W.resid) E::unpack(__ldg(reinterpret_cast<const uint4 *>(rd + off)), fd);
#pragma unroll
            for (int j = 0; j < VE; ++j) sum = __fadd_rn(sum, W(ft[j], W.resid ? fd[j] : 0.f));
          }
        } else {
          for (int e = e0; e < e1; ++e)
            sum = __fadd_rn(sum, W(E::load(rt, lo + e), W.resid ? E::load(rd, lo + e) : 0.f));
        }
        float total;
        excl = block_exclusive_scan(sum, sh.fscratch, &total);
        if (tid < static_cast<int>(C)) dsmem_st_f32(dsmem_addr(&sh.xz[par][round][rank], tid), total);
        cluster_sync();  // slice masses visible cluster-wide
        if (tid == 0) {
          float Z = 0.f;
          for (uint32_t r = 0; r < C; ++r) Z += sh.xz[par][round][r];
          int again = 0;
          if (W.resid && !(Z > 0.f)) {
            again = 1;  // no residual mass in fp32: draw from p at this position
          } else {
            const uint32_t pos = static_cast<uint32_t>(pair ? i : p.K);
            const float t = philox_uniform(p.seed, static_cast<uint32_t>(b), pos, 1u) * Z;
            float P = 0.f, Pown = 0.f, Plast = 0.f;
            int own = -1, last = -1;
            for (uint32_t r = 0; r < C; ++r) {
              const float zr = sh.xz[par][round][r];
              if (own < 0 && P + zr > t) {
                own = static_cast<int>(r);
                Pown = P;
              }
              if (zr > 0.f) {
                last = static_cast<int>(r);
                Plast = P;
              }
              P += zr;
            }
            int lastmode = 0;
            if (own < 0) {
              own = last < 0 ? 0 : last;
              Pown = Plast;
              lastmode = 1;
            }
            sh.bi[1] = own;
            sh.bi[2] = lastmode;
            sh.bf[4] = t - Pown;
          }
          sh.bi[3] = again;
        }
        __syncthreads();
        if (sh.bi[3] && round == 0) {
          W.resid = false;
          fallback = 1;
          continue;
        }
        owner = sh.bi[1];
        pl = sh.bi[2];
        tl = sh.bf[4];
        break;
      }
      taker = owner;
      if (static_cast<int>(rank) == owner) {
        // the thread whose chunk holds the crossing (or the last positive one)
        int who;
        if (!pl)
          who = block_reduce_min_int((sum > 0.f && __fadd_rn(excl, sum) > tl) ? tid : INT_MAX,
                                     sh.scratch);
        else
          who = block_reduce_max_int(sum > 0.f ? tid : -1, sh.scratch);
        if (who == INT_MAX || who < 0) {
          // rounding left no crossing in this slice: last positive entry
          pl = 1;
          who = block_reduce_max_int(sum > 0.f ? tid : -1, sh.scratch);
          if (who < 0) who = 0;
        }
        // the whole CTA walks the chosen chunk: one entry per thread, a block
        // scan, and the first entry whose running mass passes tl
        const int w0 = min(len, who * E2), w1 = min(len, w0 + E2);
        const float wexcl = __shfl_sync(0xFFFFFFFFu, excl, who & 31);
        if ((tid & 31) == 0) sh.fscratch[tid >> 5] = wexcl;
        __syncthreads();
        const float base = sh.fscratch[who >> 5];
        __syncthreads();
        float w = 0.f;
        const int e = w0 + tid;
        if (e < w1) w = W(E::load(rt, lo + e), W.resid ? E::load(rd, lo + e) : 0.f);
        float tot_unused;
        const float before = block_exclusive_scan(w, sh.fscratch, &tot_unused);
        const float run = __fadd_rn(base, __fadd_rn(before, w));
        int pick = INT_MAX;
        if (!pl) pick = block_reduce_min_int((w > 0.f && run > tl) ? e : INT_MAX, sh.scratch);
        if (pick == INT_MAX) pick = block_reduce_max_int(w > 0.f ? e : -1, sh.scratch);
        if (pick < 0) pick = w0;
        if (tid == 0) {
          p.cand[static_cast<size_t>(b) * p.J + i] = (lo + pick) | (fallback ? CAND_FALLBACK : 0);
          __threadfence();
        }
      }
    }
    if (static_cast<int>(rank) == taker) {
      if (take_ticket(p, b, sh)) emit_chain_sample(p, b);
    }
  }
  if (st.timed_out) {
    atomicOr(p.status, ST_TIMEOUT);
    st.drain_after_timeout(seq);
  }
  // keep this CTA's shared memory alive until no peer can read it
  cluster_sync();
}

// ======================================================================
// Greedy chain (T = 0) and greedy tree: per-row argmax, then the walk.
// ======================================================================
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT, 3) argmax_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ SharedSmall sh;

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();

  Stream<DT, TMA> st;
  st.p = &p;
  st.buf = dyn;
  st.full = sh.full;
  st.cl = blockIdx.x / C;
  st.lo = static_cast<int>(rank) * p.slice;
  st.len = max(0, min(p.V, st.lo + p.slice) - st.lo);
  st.nt = (st.len + p.tile - 1) / p.tile;
  st.S = p.stages;
  st.srows = 1;
  st.timed_out = false;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  st.prologue();

  int seq = 0;
  for (int n = 0;; ++n) {
    const int q = st.cl + n * p.ncl;
    if (q >= p.njobs) break;
    const int par = n & 1;
    int b, i;
    decode_job(p, q, b, i);
    const unsigned char *rt, *rd;
    st.rows_of(q, rt, rd);

    float best = -INFINITY;
    int bidx = INT_MAX;
    for (int k = 0; k < st.nt; ++k, ++seq) {
      st.acquire(seq, k, rt, nullptr);
      const int s = seq % st.S;
      const int nv = (st.tile_len(k) + VE - 1) / VE;
      const unsigned char *bt = st.stage_row(s, 0);
      const int base = st.lo + k * p.tile;
      for (int j = tid; j < nv; j += NT) {
        float f[VE];
        E::unpack(lds128(bt + j * 16), f);
        float vm = f[0];
#pragma unroll
        for (int e = 1; e < VE; ++e) vm = fmaxf(vm, f[e]);
        if (vm > best) {  // rare after the first few vectors
          best = vm;
#pragma unroll
          for (int e = VE - 1; e >= 0; --e)
            if (f[e] == vm) bidx = base + j * VE + e;
        }
      }
      st.release(seq);
    }
    block_reduce_argmax(best, bidx, sh.fscratch, sh.scratch);
    if (tid == 0)  // push this slice's (max, index) into rank 0
      dsmem_st_v4f32(dsmem_addr(&sh.xs[par][rank][0], 0), best, __int_as_float(bidx), 0.f, 0.f);
    cluster_sync();  // partial maxima of job n visible cluster-wide
    if (rank != 0) continue;
    if (tid == 0) {
      float v = -INFINITY;
      int idx = INT_MAX;
      for (uint32_t r = 0; r < C; ++r) am_combine(v, idx, sh.xs[par][r][0], __float_as_int(sh.xs[par][r][1]));
      if (idx == INT_MAX) idx = 0;  // every logit is -inf: first index
      p.cand[static_cast<size_t>(b) * p.J + i] = idx;
      if (p.kind == KIND_GREEDY_CHAIN) {
        const int R = 2 * p.K + 1;
        if (p.out_row_max) {
          p.out_row_max[static_cast<size_t>(b) * R + i] = v;
          if (i < p.K) p.out_row_max[static_cast<size_t>(b) * R + p.K + 1 + i] = NAN;
        }
        if (p.out_row_sumexp) {
          p.out_row_sumexp[static_cast<size_t>(b) * R + i] = NAN;
          if (i < p.K) p.out_row_sumexp[static_cast<size_t>(b) * R + p.K + 1 + i] = NAN;
        }
      }
    }
    if (!take_ticket(p, b, sh)) continue;

    // ---- emission: every row of sequence b has its argmax in cand[b, :]
    int *s_amax = reinterpret_cast<int *>(dyn + p.emit_off);
    int *s_tok = s_amax + p.J;
    for (int e = tid; e < p.J; e += NT) s_amax[e] = __ldcg(p.cand + static_cast<size_t>(b) * p.J + e);
    if (p.kind == KIND_GREEDY_CHAIN) {
      for (int e = tid; e < p.K; e += NT) s_tok[e] = __ldg(p.tokens + static_cast<size_t>(b) * p.K + e);
      __syncthreads();
      if (tid == 0) {
        int nacc = p.K, err = 0;
        for (int e = 0; e < p.K; ++e) {
          const int x = s_tok[e];
          if (x < 0 || x >= p.V) err = 1;
          if (nacc == p.K && x != s_amax[e]) nacc = e;
        }
        int32_t *out = p.out_tokens + static_cast<size_t>(b) * (p.K + 1);
        for (int e = 0; e <= p.K; ++e)
          out[e] = err ? -1 : (e < nacc ? s_tok[e] : (e == nacc ? s_amax[nacc] : -1));
        p.out_n[b] = err ? -1 : nacc;
        if (err) atomicOr(p.status, ST_TOKEN);
        if (p.stats) {
          if (err) {
            atomicAdd(&p.stats->errors, 1ull);
          } else {
            atomicAdd(&p.stats->sequences, 1ull);
            atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(nacc));
            atomicAdd(nacc == p.K ? &p.stats->bonus : &p.stats->resampled, 1ull);
          }
        }
        p.ticket[b] = 0;
      }
      __syncthreads();
      continue;
    }

    // tree: N = J nodes
    const int N = p.J;
    int *s_par = s_tok + N;
    int *s_depth = s_par + N;
    unsigned char *s_acc = reinterpret_cast<unsigned char *>(s_depth + N);
    for (int e = tid; e < N; e += NT) {
      s_tok[e] = __ldg(p.tokens + static_cast<size_t>(b) * N + e);
      s_par[e] = __ldg(p.parent + e);
    }
    __syncthreads();
    if (tid == 0) {
      const int W = p.max_depth + 1;
      int32_t *path = p.out_tokens + static_cast<size_t>(b) * W;
      int bad_parent = s_par[0] != -1, bad_tok = 0;
      s_depth[0] = 0;
      s_acc[0] = 1;
      int bestn = 0;
      for (int c2 = 1; c2 < N && !bad_parent; ++c2) {
        const int pc = s_par[c2];
        if (pc < 0 || pc >= c2) {
          bad_parent = 1;
          break;
        }
        const int d = s_depth[pc] + 1;
        if (d > p.max_depth) {
          bad_parent = 1;
          break;
        }
        const int x = s_tok[c2];
        if (x < 0 || x >= p.V) bad_tok = 1;
        s_depth[c2] = d;
        s_acc[c2] = s_acc[pc] && x == s_amax[pc];
        if (s_acc[c2] && d > s_depth[bestn]) bestn = c2;
      }
      if (bad_parent || bad_tok) {
        for (int e = 0; e < W; ++e) path[e] = -1;
        p.out_n[b] = -1;
        atomicOr(p.status, bad_parent ? ST_PARENT : ST_TOKEN);
      } else {
        const int d = s_depth[bestn];
        for (int e = d + 1; e < W; ++e) path[e] = -1;
        path[d] = s_amax[bestn];
        for (int n2 = bestn, e = d - 1; n2 != 0; n2 = s_par[n2], --e) path[e] = s_tok[n2];
        p.out_n[b] = d + 1;
      }
      p.ticket[b] = 0;
    }
    __syncthreads();
  }
  if (st.timed_out) {
    atomicOr(p.status, ST_TIMEOUT);
    st.drain_after_timeout(seq);
  }
  cluster_sync();
}

// ======================================================================
// Tree-attention mask and depth position IDs, one CTA per tree.
// ======================================================================
__global__ void __launch_bounds__(NT) tree_mask_kernel(const int32_t *parent, int N, int W,
                                                       uint32_t *out_mask, int32_t *out_depth,
                                                       int32_t *status) {
  __shared__ int s_bad;
  const int b = blockIdx.x;
  const int32_t *par = parent + static_cast<size_t>(b) * N;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += NT) {
    const int pn = __ldg(par + n);
    if ((n == 0 && pn != -1) || (n > 0 && (pn < 0 || pn >= n))) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  const int bad = s_bad;
  if (bad && threadIdx.x == 0) atomicOr(status, ST_PARENT);
  for (int n = threadIdx.x; n < N; n += NT) {
    uint32_t *row = out_mask + (static_cast<size_t>(b) * N + n) * W;
    for (int w = 0; w < W; ++w) row[w] = 0u;
    if (bad) {
      out_depth[static_cast<size_t>(b) * N + n] = -1;
      continue;
    }
    int depth = 0;
    for (int a = n; a != -1; a = __ldg(par + a)) {  // parent[a] < a: terminates
      row[a >> 5] |= 1u << (a & 31);
      if (a != n) ++depth;
    }
    out_depth[static_cast<size_t>(b) * N + n] = depth;
  }
}

}  // namespace spec
