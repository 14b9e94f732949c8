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
  int stages;               // shared-memory stages
  int resident;             // 1: every tile of a slice stays in shared memory
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

// Exclusive prefix sum over the threads of the block, in thread order.
__device__ __forceinline__ float block_exclusive_scan(float v, float *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float n = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc += n;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  float base = 0.f;
  for (int w = 0; w < warp; ++w) base += sh[w];
  __syncthreads();
  return base + inc - v;
}

// -------------------------------------------------------- tile pipeline
// Streams the tiles of one CTA's vocabulary slice (1 or 2 rows) through a
// ring of shared-memory stages.  TMA path: thread 0 issues one bulk copy per
// row and tile, completion is tracked by one mbarrier per stage.  Plain path
// (rows not 16-byte aligned): all threads copy element by element and pad
// the last vector with -inf.
template <int DT, bool TMA>
struct Pipe {
  using E = Elem<DT>;
  unsigned char *buf;
  uint64_t *full;
  const unsigned char *src[2];  // row bytes at the slice start
  int nrows, stages, tile, len, ntile;
  uint32_t parity;
  bool timed_out;

  __device__ __forceinline__ int tile_len(int k) const { return min(tile, len - k * tile); }
  __device__ __forceinline__ unsigned char *stage_row(int s, int r) const {
    return buf + static_cast<size_t>(s * nrows + r) * tile * E::BYTES;
  }

  // TMA only, thread 0 only.
  __device__ __forceinline__ void issue(int k, int s) {
    const uint32_t bytes = static_cast<uint32_t>(tile_len(k)) * E::BYTES;
    mbar_arrive_expect_tx(&full[s], bytes * nrows);
    for (int r = 0; r < nrows; ++r)
      bulk_g2s(stage_row(s, r), src[r] + static_cast<size_t>(k) * tile * E::BYTES, bytes, &full[s]);
  }

  __device__ __forceinline__ void prologue() {
    if (TMA && threadIdx.x == 0) {
      const int n = min(stages, ntile);
      for (int k = 0; k < n; ++k) issue(k, k);
    }
  }

  // Makes tile k available in stage s (called by every thread).
  __device__ __forceinline__ void acquire(int k, int s) {
    if (TMA) {
      const uint32_t par = (parity >> s) & 1u;
      if (!mbar_try_wait(&full[s], par)) {
        const uint64_t t0 = clock_ns();
        while (!mbar_try_wait(&full[s], par)) {
          if (clock_ns() - t0 > WAIT_LIMIT_NS) {
            timed_out = true;
            break;
          }
        }
      }
      parity ^= 1u << s;
    } else {
      __syncthreads();
      const int n = tile_len(k);
      const int npad = (n + E::VE - 1) / E::VE * E::VE;
      for (int r = 0; r < nrows; ++r) {
        const unsigned char *g = src[r] + static_cast<size_t>(k) * tile * E::BYTES;
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

  // After consuming tile k from stage s: refill the stage with tile k + stages.
  __device__ __forceinline__ void release(int k, int s) {
    if (TMA && k + stages < ntile) {
      __syncthreads();
      if (threadIdx.x == 0) issue(k + stages, s);
    }
  }

  // Bounded drain of copies that may still be in flight after a timeout.
  __device__ __forceinline__ void drain_after_timeout() {
    if (!TMA) return;
    const uint64_t t0 = clock_ns();
    for (int s = 0; s < stages; ++s)
      while (!mbar_try_wait(&full[s], (parity >> s) & 1u) && clock_ns() - t0 < WAIT_LIMIT_NS) {
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

// --------------------------------------------------------- shared state
struct SharedSmall {
  uint64_t full[MAX_STAGES];
  float red_m[2][NWARP];
  float red_s[2][NWARP];
  float part[6];      // exchanged through DSMEM: m_t, s_t, m_d, s_d, hint (int bits), argmax idx
  float zpart[2];     // exchanged: residual / fallback mass of this CTA's slice
  int tok;            // rank 0: the drawn token
  float tsum[MAX_TILES];
  float f[8];
  int i[8];
  int scratch[NWARP];
  float fscratch[NWARP];
};

// Emission by the last job of sequence b (rank 0 CTA of that cluster).
// Returns true in every thread of the CTA if this CTA is the last.
__device__ __forceinline__ bool take_ticket(const Params &p, int b, SharedSmall &sh) {
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&p.ticket[b], 1);
    sh.i[7] = (old == p.J - 1);
    if (old == p.J - 1) __threadfence();
  }
  __syncthreads();
  return sh.i[7] != 0;
}

// ======================================================================
// Stochastic chain: rows statistics, acceptance test, residual/bonus draw.
// ======================================================================
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT) sample_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  constexpr int CH = VE * VECS_PER_THREAD;  // contiguous elements per thread in a tile scan
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ SharedSmall sh;

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const int job = blockIdx.x / C;
  const int b = job / p.J;
  const int i = job - b * p.J;
  const bool pair = i < p.K;
  const float c = p.c;

  const int lo = static_cast<int>(rank) * p.slice;
  const int len = max(0, min(p.V, lo + p.slice) - lo);

  const unsigned char *rowt = static_cast<const unsigned char *>(p.zt) +
                              (static_cast<size_t>(b) * p.J + i) * p.V * E::BYTES;
  const unsigned char *rowd =
      pair ? static_cast<const unsigned char *>(p.zd) + (static_cast<size_t>(b) * p.K + i) * p.V * E::BYTES
           : nullptr;

  Pipe<DT, TMA> pipe;
  pipe.buf = dyn;
  pipe.full = sh.full;
  pipe.src[0] = rowt + static_cast<size_t>(lo) * E::BYTES;
  pipe.src[1] = pair ? rowd + static_cast<size_t>(lo) * E::BYTES : nullptr;
  pipe.nrows = pair ? 2 : 1;
  pipe.stages = p.stages;
  pipe.tile = p.tile;
  pipe.len = len;
  pipe.ntile = (len + p.tile - 1) / p.tile;
  pipe.parity = 0;
  pipe.timed_out = false;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pipe.prologue();

  // gather the draft token's two logits (another warp, overlapping the copies)
  if (tid == 32 || (NT <= 32 && tid == 0)) {
    int ok = 1, x = 0;
    float zx_t = 0.f, zx_d = 0.f;
    if (pair) {
      x = __ldg(p.tokens + static_cast<size_t>(b) * p.K + i);
      ok = (x >= 0 && x < p.V);
      if (ok) {
        zx_t = E::load(rowt, x);
        zx_d = E::load(rowd, x);
      }
    }
    sh.i[0] = ok;
    sh.f[0] = zx_t;
    sh.f[1] = zx_d;
    // hint: lowest rejected position already published for this sequence
    if (rank == 0) {
      const int hint = *reinterpret_cast<volatile int *>(p.first_rej + b);
      sh.part[4] = __int_as_float(hint);
    }
  }

  // ---- pass 1: online max / sum-exp of the slice, both rows at once
  float mt = -INFINITY, st = 0.f, mtc = 0.f;
  float md = -INFINITY, sd = 0.f, mdc = 0.f;
  for (int k = 0; k < pipe.ntile; ++k) {
    const int s = k % p.stages;
    pipe.acquire(k, s);
    const int nv = (pipe.tile_len(k) + VE - 1) / VE;
    const unsigned char *bt = pipe.stage_row(s, 0);
    if (pair) {
      const unsigned char *bd = pipe.stage_row(s, 1);
      for (int j = tid; j < nv; j += NT) {
        float f[VE];
        E::unpack(lds128(bt + j * 16), f);
        online_update<VE>(f, c, mt, st, mtc);
        E::unpack(lds128(bd + j * 16), f);
        online_update<VE>(f, c, md, sd, mdc);
      }
    } else {
      for (int j = tid; j < nv; j += NT) {
        float f[VE];
        E::unpack(lds128(bt + j * 16), f);
        online_update<VE>(f, c, mt, st, mtc);
      }
    }
    if (!p.resident) pipe.release(k, s);
  }
  block_reduce_ms(mt, st, c, sh.red_m[0], sh.red_s[0]);
  if (pair) block_reduce_ms(md, sd, c, sh.red_m[1], sh.red_s[1]);
  if (tid == 0) {
    sh.part[0] = mt;
    sh.part[1] = st;
    sh.part[2] = md;
    sh.part[3] = sd;
  }
  cluster_sync();  // #1: partial statistics visible cluster-wide

  // ---- combine the slices (rank order) and take the acceptance decision
  if (tid == 0) {
    float Mt = -INFINITY, St = 0.f, Md = -INFINITY, Sd = 0.f;
    for (uint32_t r = 0; r < C; ++r) {
      ms_combine(Mt, St, dsmem_ld_f32(dsmem_addr(&sh.part[0], r)),
                 dsmem_ld_f32(dsmem_addr(&sh.part[1], r)), c);
      if (pair)
        ms_combine(Md, Sd, dsmem_ld_f32(dsmem_addr(&sh.part[2], r)),
                   dsmem_ld_f32(dsmem_addr(&sh.part[3], r)), c);
    }
    const int hint = __float_as_int(dsmem_ld_f32(dsmem_addr(&sh.part[4], 0)));
    const int ok = sh.i[0];
    int accept = 1;
    if (pair && ok) {
      const float a = fmaf(sh.f[0], c, -(Mt * c));
      const float d = fmaf(sh.f[1], c, -(Md * c));
      const float ratio = ex2(a - d) * (Sd / St);  // p_i(x_i) / q_i(x_i)
      const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u);
      accept = u < ratio;
    }
    const int need = pair ? (ok && !accept) : 1;
    const int superseded = pair ? (hint < i) : (hint < p.K);
    sh.i[1] = accept;
    sh.i[2] = need && !superseded;
    sh.f[2] = Mt;
    sh.f[3] = St;
    sh.f[4] = Md;
    sh.f[5] = Sd;
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
  const int do_draw = sh.i[2];
  const float Mt = sh.f[2], St = sh.f[3], Md = sh.f[4], Sd = sh.f[5];
  const float mtc_g = Mt * c, mdc_g = Md * c;
  const float inv_st = 1.f / St, inv_sd = 1.f / Sd;

  // ---- pass 2 (only for a reject or the bonus row): weights, slice mass,
  // owner slice and tile, then a block scan inside the owner tile.
  int fallback = 0;
  if (do_draw) {
    // weights: residual max(0, p - q) on a pair, p (unnormalised) otherwise
    bool resid = pair;
    float t_local = 0.f;
    int owner = 0, pick_last = 0;
    for (int round = 0; round < 2; ++round) {
      if (!p.resident) {
        __syncthreads();
        pipe.prologue();
      }
      for (int k = 0; k < pipe.ntile; ++k) {
        const int s = k % p.stages;
        if (!p.resident) pipe.acquire(k, s);
        const int nv = (pipe.tile_len(k) + VE - 1) / VE;
        float acc = 0.f;
        const unsigned char *bt = pipe.stage_row(s, 0);
        if (resid) {
          const unsigned char *bd = pipe.stage_row(s, 1);
          for (int j = tid; j < nv; j += NT) {
            float ft[VE], fd[VE];
            E::unpack(lds128(bt + j * 16), ft);
            E::unpack(lds128(bd + j * 16), fd);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              const float w = ex2(fmaf(ft[e], c, -mtc_g)) * inv_st - ex2(fmaf(fd[e], c, -mdc_g)) * inv_sd;
              acc += fmaxf(w, 0.f);
            }
          }
        } else {
          for (int j = tid; j < nv; j += NT) {
            float ft[VE];
            E::unpack(lds128(bt + j * 16), ft);
#pragma unroll
            for (int e = 0; e < VE; ++e) acc += ex2(fmaf(ft[e], c, -mtc_g));
          }
        }
        const float tsum = block_reduce_sum(acc, sh.fscratch);
        if (tid == 0) sh.tsum[k] = tsum;
        if (!p.resident) pipe.release(k, s);
      }
      if (tid == 0) {
        float z = 0.f;
        for (int k = 0; k < pipe.ntile; ++k) z += sh.tsum[k];
        sh.zpart[round] = z;
      }
      cluster_sync();  // #2: slice masses visible cluster-wide
      if (tid == 0) {
        float Z = 0.f;
        for (uint32_t r = 0; r < C; ++r) Z += dsmem_ld_f32(dsmem_addr(&sh.zpart[round], r));
        int again = 0;
        if (resid && !(Z > 0.f)) {
          again = 1;  // no residual mass in fp32: draw from p at this position
        } else {
          const uint32_t pos = static_cast<uint32_t>(pair ? i : p.K);
          const float t = philox_uniform(p.seed, static_cast<uint32_t>(b), pos, 1u) * Z;
          float P = 0.f, Pown = 0.f, Plast = 0.f;
          int own = -1, last = -1;
          for (uint32_t r = 0; r < C; ++r) {
            const float zr = dsmem_ld_f32(dsmem_addr(&sh.zpart[round], r));
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
          int pl = 0;
          if (own < 0) {
            own = last < 0 ? 0 : last;
            Pown = Plast;
            pl = 1;
          }
          sh.i[3] = own;
          sh.i[4] = pl;
          sh.f[6] = t - Pown;
        }
        sh.i[5] = again;
      }
      __syncthreads();
      if (sh.i[5] && round == 0) {
        resid = false;
        fallback = 1;
        continue;
      }
      owner = sh.i[3];
      pick_last = sh.i[4];
      t_local = sh.f[6];
      break;
    }

    if (static_cast<int>(rank) == owner) {
      // owner tile: first tile whose running mass passes t_local
      if (tid == 0) {
        float TP = 0.f, TPk = 0.f, TPlast = 0.f;
        int kk = -1, klast = -1;
        for (int k = 0; k < pipe.ntile; ++k) {
          const float ts = sh.tsum[k];
          if (kk < 0 && TP + ts > t_local) {
            kk = k;
            TPk = TP;
          }
          if (ts > 0.f) {
            klast = k;
            TPlast = TP;
          }
          TP += ts;
        }
        int pl = pick_last;
        if (pl || kk < 0) {
          kk = klast < 0 ? 0 : klast;
          TPk = TPlast;
          pl = 1;
        }
        sh.i[3] = kk;
        sh.i[4] = pl;
        sh.f[6] = t_local - TPk;
      }
      __syncthreads();
      const int kk = sh.i[3];
      const int pl = sh.i[4];
      const float tl = sh.f[6];
      int s = kk;
      if (!p.resident) {
        __syncthreads();
        s = 0;
        if (TMA && tid == 0) pipe.issue(kk, 0);
        pipe.acquire(kk, 0);
      }
      const int n = pipe.len > 0 ? pipe.tile_len(kk) : 0;
      // contiguous chunk of this thread inside the tile
      const int e0 = tid * CH;
      float w[CH];
      float sum = 0.f;
      const unsigned char *bt = pipe.stage_row(s, 0);
      const unsigned char *bd = resid ? pipe.stage_row(s, 1) : nullptr;
#pragma unroll
      for (int v = 0; v < VECS_PER_THREAD; ++v) {
        const int base = e0 + v * VE;
        float ft[VE], fd[VE];
        if (base < n) {
          E::unpack(lds128(bt + base * E::BYTES), ft);
          if (resid) E::unpack(lds128(bd + base * E::BYTES), fd);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          float x = 0.f;
          if (base + e < n) {
            if (resid)
              x = fmaxf(ex2(fmaf(ft[e], c, -mtc_g)) * inv_st - ex2(fmaf(fd[e], c, -mdc_g)) * inv_sd, 0.f);
            else
              x = ex2(fmaf(ft[e], c, -mtc_g));
          }
          w[v * VE + e] = x;
          sum += x;
        }
      }
      const float excl = block_exclusive_scan(sum, sh.fscratch);
      int pick = INT_MAX;
      if (!pl) {
        float run = excl;
#pragma unroll
        for (int e = 0; e < CH; ++e) {
          run += w[e];
          if (pick == INT_MAX && run > tl && w[e] > 0.f) pick = e0 + e;
        }
      }
      pick = block_reduce_min_int(pick, sh.scratch);
      if (pick == INT_MAX) {
        int lastpos = -1;
#pragma unroll
        for (int e = 0; e < CH; ++e)
          if (w[e] > 0.f) lastpos = e0 + e;
        pick = block_reduce_max_int(lastpos, sh.scratch);
        if (pick < 0) pick = 0;
      }
      if (tid == 0) dsmem_st_s32(dsmem_addr(&sh.tok, 0), lo + kk * p.tile + pick);
    }
  }
  cluster_sync();  // #3: token delivered to rank 0; no DSMEM access after this
  if (pipe.timed_out) {
    atomicOr(p.status, ST_TIMEOUT);
    pipe.drain_after_timeout();
  }
  if (rank != 0) return;
  if (tid == 0 && do_draw) p.cand[static_cast<size_t>(b) * p.J + i] = sh.tok | (fallback ? CAND_FALLBACK : 0);

  // ---- emission by the last job of the sequence
  if (!take_ticket(p, b, sh)) return;
  const int err = __ldcg(p.seq_err + b);
  const int n = min(__ldcg(p.first_rej + b), p.K);
  for (int e = tid; e <= p.K; e += NT) {
    int v = -1;
    if (!err) {
      if (e < n)
        v = __ldg(p.tokens + static_cast<size_t>(b) * p.K + e);
      else if (e == n)
        v = __ldcg(p.cand + static_cast<size_t>(b) * p.J + n) & ~CAND_FALLBACK;
    }
    p.out_tokens[static_cast<size_t>(b) * (p.K + 1) + e] = v;
  }
  if (tid == 0) {
    p.out_n[b] = err ? -1 : n;
    if (p.stats) {
      if (err) {
        atomicAdd(&p.stats->errors, 1ull);
      } else {
        atomicAdd(&p.stats->sequences, 1ull);
        atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(n));
        if (n == p.K)
          atomicAdd(&p.stats->bonus, 1ull);
        else
          atomicAdd(&p.stats->resampled, 1ull);
        if (n < p.K && (__ldcg(p.cand + static_cast<size_t>(b) * p.J + n) & CAND_FALLBACK))
          atomicAdd(&p.stats->residual_fallbacks, 1ull);
      }
    }
    p.ticket[b] = 0;
    p.first_rej[b] = FIRST_REJ_NONE;
    p.seq_err[b] = 0;
  }
}

// ======================================================================
// Greedy chain (T = 0) and greedy tree: per-row argmax, then the walk.
// ======================================================================
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT) argmax_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ SharedSmall sh;

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const uint32_t C = cluster_size();
  const int job = blockIdx.x / C;
  const int b = job / p.J;
  const int i = job - b * p.J;
  const int lo = static_cast<int>(rank) * p.slice;
  const int len = max(0, min(p.V, lo + p.slice) - lo);
  const unsigned char *row = static_cast<const unsigned char *>(p.zt) +
                             (static_cast<size_t>(b) * p.J + i) * p.V * E::BYTES;

  Pipe<DT, TMA> pipe;
  pipe.buf = dyn;
  pipe.full = sh.full;
  pipe.src[0] = row + static_cast<size_t>(lo) * E::BYTES;
  pipe.src[1] = nullptr;
  pipe.nrows = 1;
  pipe.stages = p.stages;
  pipe.tile = p.tile;
  pipe.len = len;
  pipe.ntile = (len + p.tile - 1) / p.tile;
  pipe.parity = 0;
  pipe.timed_out = false;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pipe.prologue();

  float best = -INFINITY;
  int bidx = INT_MAX;
  for (int k = 0; k < pipe.ntile; ++k) {
    const int s = k % p.stages;
    pipe.acquire(k, s);
    const int nv = (pipe.tile_len(k) + VE - 1) / VE;
    const unsigned char *bt = pipe.stage_row(s, 0);
    const int base = lo + k * p.tile;
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
    pipe.release(k, s);
  }
  block_reduce_argmax(best, bidx, sh.fscratch, sh.scratch);
  if (tid == 0) {
    sh.part[0] = best;
    sh.part[5] = __int_as_float(bidx);
  }
  cluster_sync();  // #1
  if (rank == 0 && tid == 0) {
    float v = -INFINITY;
    int idx = INT_MAX;
    for (uint32_t r = 0; r < C; ++r)
      am_combine(v, idx, dsmem_ld_f32(dsmem_addr(&sh.part[0], r)),
                 __float_as_int(dsmem_ld_f32(dsmem_addr(&sh.part[5], r))));
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
  cluster_sync();  // #2: no DSMEM access after this
  if (pipe.timed_out) {
    atomicOr(p.status, ST_TIMEOUT);
    pipe.drain_after_timeout();
  }
  if (rank != 0) return;
  if (!take_ticket(p, b, sh)) return;

  // ---- emission: all rows of sequence b have their argmax in cand[b, :]
  int *s_amax = reinterpret_cast<int *>(dyn);
  int *s_tok = s_amax + p.J;
  for (int e = tid; e < p.J; e += NT) s_amax[e] = __ldcg(p.cand + static_cast<size_t>(b) * p.J + e);
  if (p.kind == KIND_GREEDY_CHAIN) {
    for (int e = tid; e < p.K; e += NT) s_tok[e] = __ldg(p.tokens + static_cast<size_t>(b) * p.K + e);
    __syncthreads();
    if (tid == 0) {
      int n = p.K, err = 0;
      for (int e = 0; e < p.K; ++e) {
        const int x = s_tok[e];
        if (x < 0 || x >= p.V) err = 1;
        if (n == p.K && x != s_amax[e]) n = e;
      }
      int32_t *out = p.out_tokens + static_cast<size_t>(b) * (p.K + 1);
      for (int e = 0; e <= p.K; ++e) out[e] = err ? -1 : (e < n ? s_tok[e] : (e == n ? s_amax[n] : -1));
      p.out_n[b] = err ? -1 : n;
      if (err) atomicOr(p.status, ST_TOKEN);
      if (p.stats) {
        if (err) {
          atomicAdd(&p.stats->errors, 1ull);
        } else {
          atomicAdd(&p.stats->sequences, 1ull);
          atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(n));
          atomicAdd(n == p.K ? &p.stats->bonus : &p.stats->resampled, 1ull);
        }
      }
      p.ticket[b] = 0;
    }
    return;
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
    int best = 0;
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
      if (s_acc[c2] && d > s_depth[best]) best = c2;
    }
    if (bad_parent || bad_tok) {
      for (int e = 0; e < W; ++e) path[e] = -1;
      p.out_n[b] = -1;
      atomicOr(p.status, bad_parent ? ST_PARENT : ST_TOKEN);
    } else {
      const int d = s_depth[best];
      for (int e = d + 1; e < W; ++e) path[e] = -1;
      path[d] = s_amax[best];
      for (int n2 = best, e = d - 1; n2 != 0; n2 = s_par[n2], --e) path[e] = s_tok[n2];
      p.out_n[b] = d + 1;
    }
    p.ticket[b] = 0;
  }
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
