// Verification kernels for sm_103a.
//
// Two launches per call on the caller's stream; the second is a programmatic
// dependent of the first, the first of whatever precedes it.
//
//  A. row_kernel — a streaming reduction over every logit row the step needs.
//     Work item = (job, vocabulary slice): a job is a target/draft row pair
//     (stochastic chain, positions i < K), the bonus target row K, or one
//     target row (greedy chain, tree).  Persistent CTAs take items from
//     sharded ticket counters and stream their tiles from HBM into shared
//     memory with TMA bulk copies (cp.async.bulk + one mbarrier per stage)
//     through a ring that runs across item boundaries.  Each consumer warp
//     ends an item with one 16-byte partial: (max, sum of 2^((z - max) log2e
//     / T)) for both rows, or (max, first index of max).  No CTA ever waits
//     for another.
//
//  B. draw_kernel (stochastic chain) — one thread-block cluster per sequence.
//     Every CTA combines the partials of all 2K+1 rows (fixed
//     order, so every CTA holds the same bits), takes the K acceptance tests,
//     and the cluster draws the single token the sequence needs: the residual
//     at the first reject, or the bonus from row K.  The residual draw
//     re-reads one row pair (L2-resident when possible) split over the
//     cluster: warp-range masses, CTA masses pushed to every CTA through
//     distributed shared memory, the owner CTA, its owner warp range, and a
//     block-wide walk of that range.  The owner CTA writes the outputs.
//
//     finish_kernel (greedy chain, tree) — one CTA per sequence: argmax per
//     row from the partials, then the left-to-right match or the tree walk.
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
constexpr int MAX_CLUSTER = 16;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s bound on any wait

// Streaming items are handed out by up to NSHARD ticket counters, one per
// 128-byte line: shard k hands out items k, k + ns, k + 2 ns, ... to the CTAs
// k, k + ns, ... of the row kernel.
constexpr int NSHARD = 32;
constexpr int TICKET_STRIDE = 32;  // ints

// device status bits (per stream)
constexpr int ST_TOKEN = 1, ST_PARENT = 2, ST_TIMEOUT = 4;

enum Kind : int { KIND_SAMPLE = 0, KIND_GREEDY_CHAIN = 1, KIND_TREE = 2, KIND_TREE_SAMPLE = 3 };
constexpr int MAX_TREE_NODES = 1024;

struct Stats {  // layout-compatible with spec_stats_t
  unsigned long long sequences, accepted, bonus, resampled, residual_fallbacks, errors, near_boundary;
};

// A decision within this relative distance of its boundary counts as near
// (the acceptance test |u - r| <= NEAR_REL max(r, 2^-24), the draw
// |t - C| <= NEAR_REL Z at either end of the drawn token's interval).
constexpr float NEAR_REL = 1e-5f;

struct Params {
  const void *zt;           // [B, J, V] target rows (J = K+1 chain, N tree)
  const void *zd;           // [B, K, V] draft rows (sampling only)
  const int32_t *tokens;    // chain: draft tokens [B, K]; tree: node tokens [B, N]
  const int32_t *parent;    // tree: [N]
  int parent_stride;        // 0: one tree for the batch; N: tree b at parent + b * N
  const int32_t *counts;    // chain: drafts of each sequence [B] in [0, K] (NULL: K)
  int point;                // chain: q is the point mass at each draft token (no draft rows)
  int B, K, V, J;           // K = drafts (chain) or N (tree)
  int kind;
  float c;                  // log2(e) / T
  uint64_t seed;
  int C;                    // vocabulary slices per row in the streaming kernel
  int slice;                // elements per slice (multiple of the vector width)
  int slice_d;              // elements per CTA in the draw (multiple of the vector width)
  int wbuf_off;             // draw: byte offset of the walk buffer in dynamic smem
  int tile;                 // elements per tile and row
  int stages;               // shared-memory stages of the tile ring
  int njobs;                // jobs in total; items = njobs * C
  int max_depth;            // tree output width - 1
  float4 *partials;         // [njobs * C * NCW], one per consumer warp
  int32_t *out_tokens;      // chain [B, K+1]; tree [B, max_depth+1]
  int32_t *out_n;           // chain n_accepted [B]; tree length [B]
  float *out_row_max;       // [B, 2K+1] or null
  float *out_row_sumexp;    // [B, 2K+1] or null
  Stats *stats;             // or null
  int32_t *status;          // device status bits
  int *tickets;             // item tickets, shard k at tickets[k * TICKET_STRIDE]; zero
                            // between calls (the decision kernel puts them back)
  int nshard;               // ticket shards in use
  unsigned long long *timer;  // measurement (or null): global-timer ns of the first row CTA's
                              // start [0], the last row CTA's end [1], the last output [2]
};

// Measurement stamps (spec_arm_timer): the earliest start and the latest end.
__device__ __forceinline__ void timer_min(const Params &p, int k) {
  if (p.timer) atomicMin(p.timer + k, static_cast<unsigned long long>(clock_ns()));
}
__device__ __forceinline__ void timer_max(const Params &p, int k) {
  if (p.timer) atomicMax(p.timer + k, static_cast<unsigned long long>(clock_ns()));
}

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
  __device__ static __forceinline__ float load_shared(const unsigned char *row, int i) {
    return reinterpret_cast<const float *>(row)[i];
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
  __device__ static __forceinline__ float load_shared(const unsigned char *row, int i) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(row)[i]) << 16);
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
// Commutative bit for bit (IEEE + and * are), so butterfly reductions give
// the same bits in every lane.
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float c) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    m = M;
    s = 0.f;
    return;
  }
  s = __fadd_rn(__fmul_rn(s, ex2((m - M) * c)), __fmul_rn(s2, ex2((m2 - M) * c)));
  m = M;
}

// Block-wide (max, sumexp) reduction; the result is valid in thread 0.
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

// (value, index) maximum with ties to the lower index; index INT_MAX = none.
// Commutative.
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

// ------------------------------------------------------------ job layout
// Job q -> (sequence b, row i).  Stochastic chain: the B bonus rows first (a
// bonus draw reads no row again), then the row pairs from position K-1 down
// to 0, so the pairs a residual draw most often re-reads (the early
// positions) are streamed last and are still in L2 when the draw runs.
// Argmax kinds: rows position-major.
__device__ __forceinline__ void decode_job(const Params &p, int q, int &b, int &i) {
  if (p.kind == KIND_SAMPLE) {
    const int k = q / p.B;  // the bonus rows first (never re-read), then pairs K-1 .. 0:
    b = q - k * p.B;         // the pairs a residual most often re-reads are streamed last
    i = k == 0 ? p.K : p.K - k;
  } else {
    i = q / p.B;
    b = q - i * p.B;
  }
}

__device__ __forceinline__ int job_of(const Params &p, int b, int i) {
  if (p.kind == KIND_SAMPLE) return (i == p.K ? 0 : p.K - i) * p.B + b;
  return i * p.B + b;
}

template <int DT>
__device__ __forceinline__ const unsigned char *target_row(const Params &p, int b, int i) {
  return static_cast<const unsigned char *>(p.zt) +
         (static_cast<size_t>(b) * p.J + i) * p.V * Elem<DT>::BYTES;
}

template <int DT>
__device__ __forceinline__ const unsigned char *draft_row(const Params &p, int b, int i) {
  return static_cast<const unsigned char *>(p.zd) +
         (static_cast<size_t>(b) * p.K + i) * p.V * Elem<DT>::BYTES;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// After the dependent-launch wait: a bounded wait of this call's streaming
// kernel (or of any earlier call on the same status word not yet read) ran
// out, so the row statistics may be incomplete; the call's outputs are then
// -1 rather than values drawn from them.
__device__ __forceinline__ bool stream_timed_out(const Params &p) {
  return (*reinterpret_cast<const volatile int32_t *>(p.status) & ST_TIMEOUT) != 0;
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ======================================================================
// A. row_kernel: streaming per-(job, slice) statistics.
// ======================================================================
// Warp-specialised: NCW consumer warps and one producer warp.  Item it =
// job * C + slice; a CTA takes items blockIdx.x, + gridDim.x, ...  The
// producer streams their tiles (up to two rows each) into a ring of `stages`
// shared-memory stages: it waits for a stage to be empty (every consumer warp
// arrived), then issues the bulk copies that complete the stage's `full`
// barrier.  Consumers wait on `full`, reduce, and arrive on `empty`.  At the
// end of an item every consumer warp writes its own 16-byte partial, so no
// barrier spans the CTA.
constexpr int NCW = 8;                  // consumer warps
constexpr int NT_ROW = (NCW + 1) * 32;  // + the producer warp

template <int DT, bool ARGMAX>
struct ItemCursor {
  using E = Elem<DT>;
  int item, lo, len, nt, nrows;
  const unsigned char *rt, *rd;
  const uint32_t *tree_internal;  // stochastic tree: bit u set iff node u has children

  __device__ __forceinline__ void set(const Params &p, int it) {
    item = it;
    nt = 0;
    if (it >= p.njobs * p.C) return;
    const int q = it / p.C, s = it - q * p.C;
    lo = s * p.slice;
    len = max(0, min(p.V, lo + p.slice) - lo);
    nt = (len + p.tile - 1) / p.tile;
    int b, i;
    decode_job(p, q, b, i);
    rt = target_row<DT>(p, b, i) + static_cast<size_t>(lo) * E::BYTES;
    const bool pair = p.kind == KIND_TREE_SAMPLE ? ((tree_internal[i >> 5] >> (i & 31)) & 1u) != 0
                                                 : (i < p.K && !p.point);
    if (!ARGMAX && pair) {
      rd = draft_row<DT>(p, b, i) + static_cast<size_t>(lo) * E::BYTES;
      nrows = 2;
    } else {
      rd = nullptr;
      nrows = 1;
    }
  }
};

// Bounded wait on an mbarrier phase; false if it ran out.  The warp sleeps
// in hardware between polls.
// Also bounded in polls (each suspends at most ~20 us), should the clock
// not advance.
constexpr int WAIT_LIMIT_POLLS = 1 << 17;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const uint64_t t0 = clock_ns();
  for (int polls = 0; !mbar_try_wait_sleep(bar, parity, 20000u); ++polls)
    if (clock_ns() - t0 > WAIT_LIMIT_NS || polls > WAIT_LIMIT_POLLS) return false;
  return true;
}

// Online (max, sum 2^((z - max) c)) state of one row in one thread; the sum
// is kept as two lanes for the packed fp32x2 adds.  mc = max(m c, -FLT_MAX)
// keeps -inf entries at weight 0 before any finite entry was seen.
struct Online {
  float m, mc;
  float2 s;
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    mc = -FLT_MAX;
    s = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ void rescale(float vm, float c) {
    if (vm > m) {
      const float r = ex2((m - vm) * c);
      s.x *= r;
      s.y *= r;
      m = vm;
      mc = fmaxf(vm * c, -FLT_MAX);
    }
  }
  // f: an even number of logits
  template <int N>
  __device__ __forceinline__ void accumulate(const float (&f)[N], float c) {
    const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      const float2 y = __ffma2_rn(make_float2(f[k], f[k + 1]), cc, nm);
      s = __fadd2_rn(s, make_float2(ex2(y.x), ex2(y.y)));
    }
  }
  __device__ __forceinline__ float sum() const { return s.x + s.y; }
};

// One 16-byte vector of logits into the online state; returns the vector's
// largest logit.
template <int DT>
__device__ __forceinline__ float online_vec16(const uint4 w, float c, Online &st) {
  float f[Elem<DT>::VE];
  Elem<DT>::unpack(w, f);
  float vm;
  if (DT == 1) {  // bf16: packed maximum of the 8 values
    const uint32_t mx = bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w));
    vm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u));
  } else {
    vm = fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
  }
  st.rescale(vm, c);
  st.accumulate(f, c);
  return vm;
}

// What the producer tells the consumers about the tile in a stage.
struct StageMeta {
  int item;   // item index, or -1: end of this CTA's stream
  int n;      // elements per row in the tile
  int nrows;  // 1 or 2
  int last;   // 1: last tile of the item
  int base;   // vocabulary index of the tile's first element (argmax)
  int pad[3];
};

// Warp-wide (max, sumexp) of per-lane online states: max butterfly, one
// rescale per lane, sum butterfly.  Every lane ends with the same bits.
__device__ __forceinline__ void warp_ms(float &m, float &s, float c) {
  float M = m;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  float t = (M == -INFINITY) ? 0.f : __fmul_rn(s, ex2((m - M) * c));
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) t = __fadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, off));
  m = M;
  s = t;
}

template <int DT, bool TMA, bool ARGMAX>
__global__ void __launch_bounds__(NT_ROW, 2) row_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  constexpr int SROWS = ARGMAX ? 1 : 2;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ uint64_t full[MAX_STAGES], empty[MAX_STAGES];
  __shared__ __align__(16) StageMeta meta[MAX_STAGES];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages;
  const float c = p.c;
  const size_t row_bytes = static_cast<size_t>(p.tile) * E::BYTES;
  auto stage_row = [&](int s, int r) -> unsigned char * {
    return dyn + (static_cast<size_t>(s) * SROWS + r) * row_bytes;
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // When launched as a dependent of the previous kernel on the stream, the
  // CTAs above were set up while that kernel finished; nothing in global
  // memory is touched before it has completed.
  pdl_wait();
  if (tid == 0) timer_min(p, 0);

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    const int nitems = p.njobs * p.C;
    ItemCursor<DT, ARGMAX> pc;
    __shared__ uint32_t tree_internal[ARGMAX ? 1 : MAX_TREE_NODES / 32];
    pc.tree_internal = tree_internal;
    if (!ARGMAX && p.kind == KIND_TREE_SAMPLE) {
      // stochastic tree: nodes with children stream their draft row too
      // (one tree per sequence: every node streams its draft row, since which
      // nodes have children differs between sequences)
      for (int w = lane; w < MAX_TREE_NODES / 32; w += 32) tree_internal[w] = p.parent_stride ? ~0u : 0u;
      __syncwarp();
      if (!p.parent_stride) {
        for (int cn = 1 + lane; cn < p.K; cn += 32) {
          const int u = __ldg(p.parent + cn);
          if (u >= 0 && u < p.K) atomicOr(&tree_internal[u >> 5], 1u << (u & 31));
        }
      }
      __syncwarp();
    }
    int pseq = 0;
    bool tmo = false;
    // every logit is streamed once: its lines are the first that L2 evicts
    const uint64_t pol = policy_evict_first();
    auto next_stage = [&]() -> int {  // wait until the next stage is free
      // Lane 0 alone waits (it alone issues the copies) and the warp learns
      // the outcome through the shuffle.  Were every lane to wait, a lane
      // polling after lane 0 had refilled the stage could find the next
      // phase complete and wait for a parity that never comes back.
      const int s = pseq % S;
      const uint32_t round = static_cast<uint32_t>(pseq / S);
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&empty[s], (round & 1u) ^ 1u);
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) tmo = true;
      return s;
    };
    // Items come from this CTA's ticket shard (the grid is a multiple of the
    // shard count, so every shard has as many CTAs as items / ns needs):
    // CTAs that run ahead take more items and all CTAs end together.  The
    // first item of CTA i is item i (no ticket, so the first copy is issued
    // at once); the shard's tickets then count from the shard's CTAs onward.
    // Lane 0 holds the next ticket, fetched one item ahead so its latency
    // hides behind the current item.
    const int ns = p.nshard;
    const int shard = static_cast<int>(blockIdx.x) % ns;
    const int per_shard = static_cast<int>(gridDim.x) / ns;
    int tk = 0;
    bool first = true;
    if (lane == 0) tk = atomicAdd(&p.tickets[shard * TICKET_STRIDE], 1) + per_shard;
    for (;;) {
      int it = nitems;
      if (lane == 0) {
        if (first) {
          it = static_cast<int>(blockIdx.x);  // the grid never exceeds the items
        } else {
          const long long cand = static_cast<long long>(tk) * ns + shard;
          if (cand < nitems) {
            it = static_cast<int>(cand);
            tk = atomicAdd(&p.tickets[shard * TICKET_STRIDE], 1) + per_shard;
          }
        }
        first = false;
      }
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      if (it >= nitems || tmo) break;
      pc.set(p, it);
      for (int k = 0; k < pc.nt; ++k, ++pseq) {
        const int s = next_stage();
        if (tmo) break;  // a wait ran out: stop (the consumers stop on their own)
        const int n = min(p.tile, pc.len - k * p.tile);
        const size_t off = static_cast<size_t>(k) * row_bytes;
        if (lane == 0) {
          StageMeta m;
          m.item = it;
          m.n = n;
          m.nrows = pc.nrows;
          m.last = (k == pc.nt - 1);
          m.base = pc.lo + k * p.tile;
          meta[s] = m;
        }
        if (TMA) {
          if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(n) * E::BYTES;
            mbar_arrive_expect_tx(&full[s], bytes * pc.nrows);
            bulk_g2s_hint(stage_row(s, 0), pc.rt + off, bytes, &full[s], pol);
            if (pc.nrows == 2) bulk_g2s_hint(stage_row(s, 1), pc.rd + off, bytes, &full[s], pol);
          }
        } else {
          const int npad = (n + VE - 1) / VE * VE;
          for (int r = 0; r < pc.nrows; ++r) {
            const unsigned char *g = (r ? pc.rd : pc.rt) + off;
            unsigned char *d = stage_row(s, r);
            for (int e = lane; e < npad; e += 32) {
              if (e < n)
                E::copy_elem(d + e * E::BYTES, g + e * E::BYTES);
              else
                E::store_neg_inf(d + e * E::BYTES);
            }
          }
          __threadfence_block();  // the lanes' copies are visible before the arrival
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
        }
      }
      if (pc.nt == 0 && lane == 0) {  // an empty slice still gets its (neutral) partials
        for (int w = 0; w < NCW; ++w)
          p.partials[static_cast<size_t>(it) * NCW + w] =
              ARGMAX ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                     : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      }
    }
    // end of stream
    const int s = next_stage();
    if (!tmo && lane == 0) {
      meta[s].item = -1;
      mbar_arrive(&full[s]);
    }
    if (tmo && lane == 0) atomicOr(p.status, ST_TIMEOUT);
    pdl_launch_dependents();
    return;
  }

  // -------------------------------------------------------------- consumers
  bool tmo = false;
  Online ot, od;  // target and draft row states
  ot.init();
  od.init();
  float av = -INFINITY;  // argmax value
  int aidx = INT_MAX;    // argmax index
  for (int seq = 0;; ++seq) {
    const int s = seq % S;
    // every lane waits (the bulk-copied bytes become visible to it); a
    // timeout ends the loop for the whole warp
    const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>(seq / S) & 1u);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      tmo = true;
      break;
    }
    const StageMeta m = meta[s];
    if (m.item < 0) break;
    // this warp's contiguous share of the tile's vectors (lanes interleaved)
    const int nv = (m.n + VE - 1) / VE;
    const int nvw = (nv + NCW - 1) / NCW;
    const int j0 = warp * nvw + lane, j1 = min(nv, (warp + 1) * nvw);
    const unsigned char *bt = stage_row(s, 0);
    if (ARGMAX) {
      for (int j = j0; j < j1; j += 32) {
        float f[VE];
        E::unpack(lds128(bt + j * 16), f);
        float vm = f[0];
#pragma unroll
        for (int e = 1; e < VE; ++e) vm = fmaxf(vm, f[e]);
        if (vm > av) {  // rare after the first few vectors
          av = vm;
#pragma unroll
          for (int e = VE - 1; e >= 0; --e)
            if (f[e] == vm) aidx = m.base + j * VE + e;
        }
      }
    } else if (m.nrows == 2) {
      const unsigned char *bd = stage_row(s, 1);
      for (int j = j0; j < j1; j += 32) {
        const uint4 wt = lds128(bt + j * 16), wd = lds128(bd + j * 16);
        online_vec16<DT>(wt, c, ot);
        online_vec16<DT>(wd, c, od);
      }
    } else {
      for (int j = j0; j < j1; j += 32) online_vec16<DT>(lds128(bt + j * 16), c, ot);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with stage s
    if (!m.last) continue;
    // end of the item: one partial per warp
    float4 out;
    if (ARGMAX) {
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, av, off);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, aidx, off);
        am_combine(av, aidx, v2, i2);
      }
      out = make_float4(av, __int_as_float(aidx), 0.f, 0.f);
      av = -INFINITY;
      aidx = INT_MAX;
    } else {
      float m_t = ot.m, s_t = ot.sum(), m_d = od.m, s_d = od.sum();
      warp_ms(m_t, s_t, c);
      if (m.nrows == 2) warp_ms(m_d, s_d, c);
      out = make_float4(m_t, s_t, m_d, s_d);
      ot.init();
      od.init();
    }
    if (lane == 0) p.partials[static_cast<size_t>(m.item) * NCW + warp] = out;
  }
  if (lane == 0) timer_max(p, 1);
  pdl_launch_dependents();
  if (tmo) atomicOr(p.status, ST_TIMEOUT);
}

// ======================================================================
// B. draw_kernel: decisions and the one draw of each sequence.
// ======================================================================
// One thread-block cluster of CD CTAs per sequence; CTA `rank` owns the
// vocabulary slice [rank * slice_d, (rank + 1) * slice_d) of the draw.
//
//  1. Before the dependent-launch wait (inputs only): the draft tokens, their
//     target and draft logits, the acceptance uniforms.
//  2. Every CTA combines the partials of all 2K+1 rows itself (the same
//     fixed order everywhere, so every CTA holds the same bits) and takes the
//     K decisions left to right: no exchange is needed for them.
//  3. n == K: rank 0 draws the bonus token from row K's partials.
//     n < K: every warp weighs a contiguous range of its CTA's slice of the
//     row pair (lane-strided, coalesced loads, several in flight per lane)
//     and sums it with shuffles; each CTA's mass goes to every CTA of the
//     cluster through distributed shared memory; after one cluster barrier
//     every CTA knows Z and the CTA holding u * Z.  That CTA finds the warp
//     range holding it, weighs the range into shared memory, and one warp
//     walks its CDF.
//
// Weight of one vocabulary entry in the draw: the residual max(0, p - q) of a
// rejected pair, or the unnormalised p of a draw from p.  Explicit roundings,
// so the summation and the walk compute identical bits.
struct Weights {
  float c, mtc, mdc, inv_st, inv_sd;
  bool resid;
  int excl;  // point-mass drafts: the rejected draft token, whose weight is 0
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float et = ex2(fmaf(zt, c, -mtc));
    if (!resid) return et;
    const float ed = ex2(fmaf(zd, c, -mdc));
    return fmaxf(__fsub_rn(__fmul_rn(et, inv_st), __fmul_rn(ed, inv_sd)), 0.f);
  }
  // Point-mass residual max(0, p - q) with q the point mass at excl: p(v)
  // rounded as fmul(et, inv_st) for v != excl (exactly the residual of a
  // one-hot draft row, whose q is 0 there), 0 at excl.
  __device__ __forceinline__ float at(float zt, float, int v) const {
    return v == excl ? 0.f : __fmul_rn(ex2(fmaf(zt, c, -mtc)), inv_st);
  }
};

struct DrawShared {
  float xz[2][MAX_CLUSTER];  // CTA masses pushed by every CTA (round 0 / 1)
  float wmass[NWARP];        // this CTA's warp-range masses
  float bf[8];
  int bi[8];
  float scan[NWARP + 1];     // block scan scratch
  int ired[NWARP];           // block reduction scratch
  int pick;                  // walk result
  float zdraw;               // the draw's total mass Z (bonus draw)
  // chain: bit i of word i / 64: position i rejected / near its boundary /
  // with a bad token (K <= 255)
  unsigned long long mrej[4], mnear[4], mbad[4];
};

constexpr int PARTS_PER_LANE = 8;

// (max, sumexp) of the target row (and of the draft row if `pair`) of one job
// from its C x NCW partials, by one warp: lane l folds partials l, l + 32, ...
// in order (PARTS_PER_LANE loads in flight per lane), then a butterfly, so
// every lane (and every CTA) ends with the same bits.
__device__ __forceinline__ void warp_norms(const float4 *parts, int nparts, float c, bool pair,
                                           float &mt, float &st, float &md, float &sd) {
  const int lane = threadIdx.x & 31;
  mt = md = -INFINITY;
  st = sd = 0.f;
  for (int base = 0; base < nparts; base += 32 * PARTS_PER_LANE) {
    float4 v[PARTS_PER_LANE];
#pragma unroll
    for (int k = 0; k < PARTS_PER_LANE; ++k) {
      const int j = base + lane + 32 * k;
      v[k] = j < nparts ? __ldcg(parts + j) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    }
#pragma unroll
    for (int k = 0; k < PARTS_PER_LANE; ++k) {
      ms_combine(mt, st, v[k].x, v[k].y, c);
      if (pair) ms_combine(md, sd, v[k].z, v[k].w, c);
    }
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float m2 = __shfl_xor_sync(0xFFFFFFFFu, mt, off), s2 = __shfl_xor_sync(0xFFFFFFFFu, st, off);
    ms_combine(mt, st, m2, s2, c);
    if (pair) {
      m2 = __shfl_xor_sync(0xFFFFFFFFu, md, off);
      s2 = __shfl_xor_sync(0xFFFFFFFFu, sd, off);
      ms_combine(md, sd, m2, s2, c);
    }
  }
}

// (max, sumexp) of the target row (and of the draft row if `pair`) of one job
// from its n partials, by one warp.  Up to 32 * JOB_PARTS_PER_LANE partials
// (all loads in flight at once): the maximum first (lane maximum, butterfly),
// one rescale per partial, then a sum butterfly; more: the partials folded
// in order.  Either way every lane (and every CTA) ends with the same bits.
constexpr int JOB_PARTS_PER_LANE = 8;
__device__ __forceinline__ void warp_job_norms(const float4 *ip, int n, float c, bool pair, float &mt,
                                               float &st, float &md, float &sd) {
  if (n > 32 * JOB_PARTS_PER_LANE) {
    warp_norms(ip, n, c, pair, mt, st, md, sd);
    return;
  }
  const int lane = threadIdx.x & 31;
  float4 v[JOB_PARTS_PER_LANE];
#pragma unroll
  for (int k = 0; k < JOB_PARTS_PER_LANE; ++k) {
    const int j = lane + 32 * k;
    v[k] = j < n ? __ldcg(ip + j) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  }
  float Mt = -INFINITY, Md = -INFINITY;
#pragma unroll
  for (int k = 0; k < JOB_PARTS_PER_LANE; ++k) {
    Mt = fmaxf(Mt, v[k].x);
    Md = fmaxf(Md, v[k].z);
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    Mt = fmaxf(Mt, __shfl_xor_sync(0xFFFFFFFFu, Mt, off));
    Md = fmaxf(Md, __shfl_xor_sync(0xFFFFFFFFu, Md, off));
  }
  float a = 0.f, d = 0.f;
#pragma unroll
  for (int k = 0; k < JOB_PARTS_PER_LANE; ++k) {
    if (Mt != -INFINITY && v[k].y != 0.f) a = __fadd_rn(a, __fmul_rn(v[k].y, ex2((v[k].x - Mt) * c)));
    if (pair && Md != -INFINITY && v[k].w != 0.f) d = __fadd_rn(d, __fmul_rn(v[k].w, ex2((v[k].z - Md) * c)));
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    a = __fadd_rn(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
    d = __fadd_rn(d, __shfl_xor_sync(0xFFFFFFFFu, d, off));
  }
  mt = Mt;
  st = a;
  md = pair ? Md : -INFINITY;
  sd = pair ? d : 0.f;
}

// Exclusive prefix sum over the lanes; *total = the warp's sum (every lane).
__device__ __forceinline__ float warp_excl_scan(float v, float *total) {
  const int lane = threadIdx.x & 31;
  float inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float n = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc = __fadd_rn(inc, n);
  }
  *total = __shfl_sync(0xFFFFFFFFu, inc, 31);
  const float ex = __shfl_up_sync(0xFFFFFFFFu, inc, 1);
  return lane ? ex : 0.f;
}

// Butterfly sum: the same bits in every lane.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

// Inverse-CDF walk of the weights wbuf[0, len) of one range whose preceding
// mass is P, by the whole CTA: the smallest entry e whose running mass
// P + C(e) passes t, else (or if `lastmode`) the last entry of positive
// weight.  Each thread holds a contiguous chunk; the chunk test and the walk
// inside the chunk compare the same sums (the chunk's prefix from zero added
// to the same base), so a chunk chosen by its total always yields an entry.
// Returns the entry index in every thread (0 if the range has no positive
// weight).
__device__ __forceinline__ int block_walk(const float *wbuf, int len, float P, float t, bool lastmode,
                                          DrawShared &sh) {
  const int tid = threadIdx.x;
  const int cper = (len + NT - 1) / NT;
  const int a0 = min(len, tid * cper), a1 = min(len, a0 + cper);
  float csum = 0.f;
  for (int e = a0; e < a1; ++e) csum = __fadd_rn(csum, wbuf[e]);
  float tot;
  const float E0 = __fadd_rn(P, block_exclusive_scan(csum, sh.scan, &tot));
  const int who = block_reduce_min_int(
      (!lastmode && csum > 0.f && __fadd_rn(E0, csum) > t) ? tid : INT_MAX, sh.ired);
  int pick = -1;
  if (who != INT_MAX) {
    if (tid == who) {
      float pre = 0.f;
      for (int e = a0; e < a1; ++e) {
        const float x = wbuf[e];
        pre = __fadd_rn(pre, x);
        if (x > 0.f && __fadd_rn(E0, pre) > t) {
          pick = e;
          break;
        }
      }
      sh.pick = pick;
    }
    __syncthreads();
    pick = sh.pick;
    __syncthreads();
  }
  if (pick < 0) {  // the last entry of positive weight
    int lastp = -1;
    for (int e = a0; e < a1; ++e)
      if (wbuf[e] > 0.f) lastp = e;
    lastp = block_reduce_max_int(lastp, sh.ired);
    pick = lastp < 0 ? 0 : lastp;
  }
  return pick;
}

// Bonus draw from p (unnormalised weights 2^((z - M) c)) of one target row,
// by one CTA, from the row's streaming partials: the partial of (slice s,
// consumer warp w) is the mass of a contiguous vocabulary range, so warp 0
// finds the range holding u * Z from the partials alone; the CTA weighs that
// range (at most one streaming tile's warp share) into `wbuf` and warp 0
// walks it.  Returns the token in thread 0.
template <int DT>
__device__ __forceinline__ int draw_p_from_partials(const Params &p, const float4 *parts,
                                                    const unsigned char *row, float M, float u,
                                                    float *wbuf, DrawShared &sh) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  const int tid = threadIdx.x, lane = tid & 31;
  const float c = p.c, Mc = M * c;
  const int nparts = p.C * NCW;
  auto mass = [&](int j) -> float {
    const float4 v = __ldcg(parts + j);
    return v.x == -INFINITY ? 0.f : __fmul_rn(v.y, ex2(fmaf(v.x, c, -Mc)));
  };
  if (tid < 32) {
    // range masses; lane l holds a contiguous run of them
    constexpr int BATCH = 4;
    const int per = (nparts + 31) / 32;
    const int j0 = min(nparts, lane * per), j1 = min(nparts, j0 + per);
    float sum = 0.f;
    for (int j = j0; j < j1; j += BATCH) {
      float v[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) v[k] = j + k < j1 ? mass(j + k) : 0.f;
#pragma unroll
      for (int k = 0; k < BATCH; ++k) sum = __fadd_rn(sum, v[k]);
    }
    float Z;
    const float excl = warp_excl_scan(sum, &Z);
    const float t = u * Z;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, sum > 0.f && __fadd_rn(excl, sum) > t);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, sum > 0.f);
    int lastmode = hit == 0;
    const int who = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == who) {
      float pre = 0.f, P = excl, Plast = excl;
      int own = -1, lastj = j0;
      for (int j = j0; j < j1; j += BATCH) {
        float v[BATCH];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) v[k] = j + k < j1 ? mass(j + k) : 0.f;
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
          const float before = __fadd_rn(excl, pre);
          pre = __fadd_rn(pre, v[k]);
          if (v[k] > 0.f) {
            if (!lastmode && own < 0 && __fadd_rn(excl, pre) > t) {
              own = j + k;
              P = before;
            }
            lastj = j + k;
            Plast = before;
          }
        }
      }
      if (own < 0) {
        own = lastj;
        P = Plast;
        lastmode = 1;
      }
      sh.bi[4] = own;
      sh.bi[5] = lastmode;
      sh.bf[4] = P;
      sh.bf[5] = t;
    }
  }
  __syncthreads();
  const int own = sh.bi[4];
  const bool lastmode = sh.bi[5] != 0;
  const float P = sh.bf[4], t = sh.bf[5];
  // the owner range: slice s, consumer warp w of the streaming split
  const int sl = own / NCW, w = own - sl * NCW;
  const int lo_s = sl * p.slice;
  const int len_s = max(0, min(p.V, lo_s + p.slice) - lo_s);
  const int nv = (len_s + VE - 1) / VE, nvw = (nv + NCW - 1) / NCW;
  const int r0 = lo_s + min(len_s, w * nvw * VE);
  const int len = lo_s + min(len_s, (w + 1) * nvw * VE) - r0;
  for (int e = tid; e < len; e += NT) wbuf[e] = ex2(fmaf(E::load(row, r0 + e), c, -Mc));
  __syncthreads();
  return r0 + block_walk(wbuf, len, P, t, lastmode, sh);
}

// This CTA's share of a cluster-wide draw: slice [lo, lo + len) of the
// vocabulary, NWARP contiguous warp ranges of nvw 16-byte vectors each.
struct DrawSlice {
  int lo, len, nv, nvw;
  __device__ __forceinline__ void set(int rank, int slice_d, int V, int VE) {
    lo = rank * slice_d;
    len = max(0, min(V, lo + slice_d) - lo);
    nv = (len + VE - 1) / VE;
    nvw = (nv + NWARP - 1) / NWARP;
  }
};

// One cluster-wide weighing of the row pair (rt, rd) under W, by every CTA
// of the cluster over its slice: each warp sums its range (lane-strided,
// coalesced 16-byte loads, four per row in flight per lane) into
// sh.wmass[warp]; each CTA's mass goes into sh.xz[slot][rank] of every CTA;
// after the cluster barrier every thread of every CTA gets the same total Z.
template <int DT, bool TMA, bool EXCL = false>
__device__ __forceinline__ float cluster_weigh(const unsigned char *rt, const unsigned char *rd, const Weights &W,
                                               const DrawSlice &ds, int slot, uint32_t rank, uint32_t CD,
                                               DrawShared &sh) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v0 = warp * ds.nvw, v1 = min(ds.nv, v0 + ds.nvw);
  float acc = 0.f;
  if (TMA) {  // rows 16-byte aligned, V a multiple of the vector width
    constexpr int BATCH = 4;
    for (int j = v0 + lane; j < v1; j += 32 * BATCH) {
      uint4 vt[BATCH], vd[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const int jj = j + 32 * k;
        const size_t off = static_cast<size_t>(ds.lo + jj * VE) * E::BYTES;
        vt[k] = jj < v1 ? __ldcg(reinterpret_cast<const uint4 *>(rt + off)) : make_uint4(0, 0, 0, 0);
        vd[k] = (jj < v1 && W.resid) ? __ldcg(reinterpret_cast<const uint4 *>(rd + off)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        if (j + 32 * k >= v1) break;
        float ft[VE], fd[VE];
        E::unpack(vt[k], ft);
        E::unpack(vd[k], fd);
#pragma unroll
        for (int e = 0; e < VE; ++e)
          acc = __fadd_rn(acc, EXCL ? W.at(ft[e], fd[e], ds.lo + (j + 32 * k) * VE + e) : W(ft[e], fd[e]));
      }
    }
  } else {
    const int e0 = min(ds.len, v0 * VE), e1 = min(ds.len, v1 * VE);
    for (int e = e0 + lane; e < e1; e += 32)
      acc = __fadd_rn(acc, EXCL ? W.at(E::load(rt, ds.lo + e), W.resid ? E::load(rd, ds.lo + e) : 0.f, ds.lo + e)
                                : W(E::load(rt, ds.lo + e), W.resid ? E::load(rd, ds.lo + e) : 0.f));
  }
  acc = warp_sum(acc);
  if (lane == 0) sh.wmass[warp] = acc;
  __syncthreads();
  if (tid < static_cast<int>(CD)) {  // this CTA's mass, into every CTA of the cluster
    float cm = 0.f;
    for (int w = 0; w < NWARP; ++w) cm = __fadd_rn(cm, sh.wmass[w]);
    dsmem_st_f32(dsmem_addr(&sh.xz[slot][rank], static_cast<uint32_t>(tid)), cm);
  }
  cluster_sync();  // every CTA's mass is in every CTA
  float Z = 0.f;
  for (uint32_t r = 0; r < CD; ++r) Z = __fadd_rn(Z, sh.xz[slot][r]);
  return Z;
}

// The CTA whose slice holds t = u * Z (the first with positive mass whose
// running total passes t; else the last with positive mass), found by
// thread 0 from sh.xz[slot]: sh.bi[2] = that CTA, sh.bi[3] = last-entry mode,
// sh.bf[0] = the mass before it, sh.bf[1] = t.  The caller synchronises.
__device__ __forceinline__ void find_owner_cta(float u, float Z, int slot, uint32_t CD, DrawShared &sh) {
  const float t = u * Z;
  float P = 0.f, Pown = 0.f, Plast = 0.f;
  int own = -1, last = -1;
  for (uint32_t r = 0; r < CD; ++r) {
    const float zr = sh.xz[slot][r];
    if (own < 0 && zr > 0.f && __fadd_rn(P, zr) > t) {
      own = static_cast<int>(r);
      Pown = P;
    }
    if (zr > 0.f) {
      last = static_cast<int>(r);
      Plast = P;
    }
    P = __fadd_rn(P, zr);
  }
  int lastmode = 0;
  if (own < 0) {
    own = last < 0 ? 0 : last;
    Pown = Plast;
    lastmode = 1;
  }
  sh.bi[2] = own;
  sh.bi[3] = lastmode;
  sh.bf[0] = Pown;
  sh.bf[1] = t;
}

// In the owner CTA (after find_owner_cta): the warp range holding t, its
// weights into wbuf (16-byte loads when the rows allow them, TMA), and the
// block-wide walk.  Returns the token in every thread.  sh.wmass must still
// hold this CTA's warp masses of the same W.
template <int DT, bool TMA, bool EXCL = false>
__device__ __forceinline__ int owner_walk(const unsigned char *rt, const unsigned char *rd, const Weights &W,
                                          const DrawSlice &ds, float *wbuf, DrawShared &sh) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  const int tid = threadIdx.x;
  if (tid == 0) {
    const float t = sh.bf[1];
    int lastmode = sh.bi[3];
    float P = sh.bf[0], Pown = P, Plast = P;
    int ow = -1, last = -1;
    for (int w = 0; w < NWARP; ++w) {
      const float m = sh.wmass[w];
      if (!lastmode && ow < 0 && m > 0.f && __fadd_rn(P, m) > t) {
        ow = w;
        Pown = P;
      }
      if (m > 0.f) {
        last = w;
        Plast = P;
      }
      P = __fadd_rn(P, m);
    }
    if (ow < 0) {
      ow = last < 0 ? 0 : last;
      Pown = Plast;
      lastmode = 1;
    }
    sh.bi[6] = ow;
    sh.bi[7] = lastmode;
    sh.bf[2] = Pown;
  }
  __syncthreads();
  const int ow = sh.bi[6];
  const int r0 = min(ds.len, ow * ds.nvw * VE);
  const int rlen = min(ds.len, (ow + 1) * ds.nvw * VE) - r0;
  if (TMA) {  // r0, rlen and the slice start are multiples of the vector width
    for (int j = tid; j < rlen / VE; j += NT) {
      const int e0 = ds.lo + r0 + j * VE;
      const size_t off = static_cast<size_t>(e0) * E::BYTES;
      const uint4 vt = __ldcg(reinterpret_cast<const uint4 *>(rt + off));
      const uint4 vd = W.resid ? __ldcg(reinterpret_cast<const uint4 *>(rd + off)) : make_uint4(0, 0, 0, 0);
      float ft[VE], fd[VE];
      E::unpack(vt, ft);
      E::unpack(vd, fd);
#pragma unroll
      for (int e = 0; e < VE; ++e) wbuf[j * VE + e] = EXCL ? W.at(ft[e], fd[e], e0 + e) : W(ft[e], fd[e]);
    }
  } else {
    for (int e = tid; e < rlen; e += NT)
      wbuf[e] = EXCL ? W.at(E::load(rt, ds.lo + r0 + e), W.resid ? E::load(rd, ds.lo + r0 + e) : 0.f, ds.lo + r0 + e)
                     : W(E::load(rt, ds.lo + r0 + e), W.resid ? E::load(rd, ds.lo + r0 + e) : 0.f);
  }
  const float Pw = sh.bf[2], tw = sh.bf[1];
  const bool lastw = sh.bi[7] != 0;
  __syncthreads();
  return ds.lo + r0 + block_walk(wbuf, rlen, Pw, tw, lastw, sh);
}

// ---------------------------------------------------------------- chain draw
// The chain's single draw weighs one row pair (a residual) or one row (a
// draw from p).  Each row's normaliser is folded into the exponent:
// p(v) = 2^(z_t(v) c - lt) with lt = m_t c + log2 S_t, and q(v) likewise, so
// a weight costs two paired FMAs and two MUFU exponentials per entry pair.
enum WMode : int { W_RESID = 0, W_P = 1, W_P_EXCL = 2 };
struct FoldedW {
  float c, lt, ld;
  int mode;  // W_RESID: max(0, p - q); W_P: p; W_P_EXCL: p, 0 at `excl`
  int excl;  // point-mass drafts: the rejected draft token
};

// Weights of the VE entries of one vector whose first entry is e0, with
// explicit roundings: every recomputation gives the same bits.
template <int VE>
__device__ __forceinline__ void vec_weights(const FoldedW &W, const float (&ft)[VE], const float (&fd)[VE],
                                            int e0, float (&w)[VE]) {
  const float2 cc = make_float2(W.c, W.c);
  const float2 nt = make_float2(-W.lt, -W.lt), nd = make_float2(-W.ld, -W.ld);
#pragma unroll
  for (int e = 0; e < VE; e += 2) {
    const float2 a = __ffma2_rn(make_float2(ft[e], ft[e + 1]), cc, nt);
    const float2 pe = make_float2(ex2(a.x), ex2(a.y));
    if (W.mode == W_RESID) {
      const float2 d = __ffma2_rn(make_float2(fd[e], fd[e + 1]), cc, nd);
      const float2 r = __ffma2_rn(make_float2(ex2(d.x), ex2(d.y)), make_float2(-1.f, -1.f), pe);  // p - q
      w[e] = fmaxf(r.x, 0.f);
      w[e + 1] = fmaxf(r.y, 0.f);
    } else {
      w[e] = (W.mode == W_P_EXCL && e0 + e == W.excl) ? 0.f : pe.x;
      w[e + 1] = (W.mode == W_P_EXCL && e0 + e + 1 == W.excl) ? 0.f : pe.y;
    }
  }
}

// Mass of one vector, summed as a pairwise tree.
template <int VE>
__device__ __forceinline__ float vec_mass(const float (&w)[VE]) {
  if constexpr (VE == 8) {
    const float2 s1 = __fadd2_rn(make_float2(w[0], w[2]), make_float2(w[1], w[3]));  // w0+w1, w2+w3
    const float2 s2 = __fadd2_rn(make_float2(w[4], w[6]), make_float2(w[5], w[7]));  // w4+w5, w6+w7
    const float2 s3 = __fadd2_rn(make_float2(s1.x, s2.x), make_float2(s1.y, s2.y));
    return __fadd_rn(s3.x, s3.y);
  } else {
    const float2 s1 = __fadd2_rn(make_float2(w[0], w[2]), make_float2(w[1], w[3]));
    return __fadd_rn(s1.x, s1.y);
  }
}

// Running masses of the entries of one vector along the same tree: pre is
// non-decreasing, an entry of weight 0 leaves it unchanged, and
// pre[VE - 1] equals vec_mass(w) bit for bit.
template <int VE>
__device__ __forceinline__ void vec_prefix(const float (&w)[VE], float (&pre)[VE]) {
  const float s01 = __fadd_rn(w[0], w[1]), s23 = __fadd_rn(w[2], w[3]);
  const float s0123 = __fadd_rn(s01, s23);
  pre[0] = w[0];
  pre[1] = s01;
  pre[2] = __fadd_rn(s01, w[2]);
  pre[3] = s0123;
  if constexpr (VE == 8) {
    const float s45 = __fadd_rn(w[4], w[5]), s67 = __fadd_rn(w[6], w[7]);
    pre[4] = __fadd_rn(s0123, w[4]);
    pre[5] = __fadd_rn(s0123, s45);
    pre[6] = __fadd_rn(s0123, __fadd_rn(s45, w[6]));
    pre[7] = __fadd_rn(s0123, __fadd_rn(s45, s67));
  }
}

// The VE logits of one vector of a row; entries at or past V read as -inf
// (weight 0).  VEC: the row is 16-byte aligned and e0 a multiple of VE.
template <int DT, bool VEC>
__device__ __forceinline__ void load_vec(const unsigned char *row, int e0, int V, float (&f)[Elem<DT>::VE]) {
  using E = Elem<DT>;
  if (VEC) {
    E::unpack(__ldcg(reinterpret_cast<const uint4 *>(row + static_cast<size_t>(e0) * E::BYTES)), f);
  } else {
#pragma unroll
    for (int e = 0; e < E::VE; ++e) f[e] = e0 + e < V ? E::load(row, e0 + e) : -INFINITY;
  }
}

// This CTA's weighing of its slice of the draw: the mass of every vector into
// wv[], each thread's sum over a contiguous chunk of vectors (cs), and a
// block-wide exclusive scan of those sums (E).  Returns the CTA's mass in
// every thread.  Loads are block-strided (coalesced) with BATCH vectors per
// row in flight per thread.
template <int DT, bool VEC>
__device__ __forceinline__ float slice_weigh(const unsigned char *rt, const unsigned char *rd, const FoldedW &W,
                                             const DrawSlice &ds, int V, float *wv, DrawShared &sh, float &E,
                                             float &cs) {
  using El = Elem<DT>;
  constexpr int VE = El::VE;
  const int tid = threadIdx.x;
  const bool pair = W.mode == W_RESID;
  if (VEC) {
    constexpr int BATCH = 4;
    for (int j0 = tid; j0 < ds.nv; j0 += NT * BATCH) {
      uint4 vt[BATCH], vd[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const int j = j0 + NT * k;
        const size_t off = static_cast<size_t>(ds.lo + j * VE) * El::BYTES;
        vt[k] = j < ds.nv ? __ldcg(reinterpret_cast<const uint4 *>(rt + off)) : make_uint4(0, 0, 0, 0);
        vd[k] = (j < ds.nv && pair) ? __ldcg(reinterpret_cast<const uint4 *>(rd + off)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const int j = j0 + NT * k;
        if (j >= ds.nv) break;
        float ft[VE], fd[VE], w[VE];
        El::unpack(vt[k], ft);
        El::unpack(vd[k], fd);
        vec_weights<VE>(W, ft, fd, ds.lo + j * VE, w);
        wv[j] = vec_mass<VE>(w);
      }
    }
  } else {
    for (int j = tid; j < ds.nv; j += NT) {
      float ft[VE], fd[VE], w[VE];
      load_vec<DT, false>(rt, ds.lo + j * VE, V, ft);
      if (pair) load_vec<DT, false>(rd, ds.lo + j * VE, V, fd);
      else
#pragma unroll
        for (int e = 0; e < VE; ++e) fd[e] = -INFINITY;
      vec_weights<VE>(W, ft, fd, ds.lo + j * VE, w);
      wv[j] = vec_mass<VE>(w);
    }
  }
  __syncthreads();
  const int cper = (ds.nv + NT - 1) / NT;
  const int a0 = min(ds.nv, tid * cper), a1 = min(ds.nv, a0 + cper);
  float s = 0.f;
  for (int j = a0; j < a1; ++j) s = __fadd_rn(s, wv[j]);
  cs = s;
  float total;
  E = block_exclusive_scan(s, sh.scan, &total);
  return total;
}

// The thread whose running mass P + E + cs first passes t (threads with
// positive mass only); if none does (rounding at the very end of the
// distribution, or lastmode), the last thread with positive mass and
// *lastmode = true.  Every thread gets the same answer.
__device__ __forceinline__ int owner_thread(float P, float t, float E, float cs, bool &lastmode, DrawShared &sh) {
  const int tid = threadIdx.x;
  int who = INT_MAX;
  if (!lastmode)
    who = block_reduce_min_int((cs > 0.f && __fadd_rn(P, __fadd_rn(E, cs)) > t) ? tid : INT_MAX, sh.ired);
  if (who == INT_MAX) {
    lastmode = true;
    who = max(0, block_reduce_max_int(cs > 0.f ? tid : -1, sh.ired));
  }
  return who;
}

// In the owner thread: the entry of vector (ft, fd, first entry e0) whose
// running mass base(pre) passes t, where base(x) = P + (E + (cbefore + x));
// else the last entry of positive weight.  Returns the entry's offset; *near
// is set when t lies within NEAR_REL Z of either end of that entry's interval.
template <int VE>
__device__ __forceinline__ int vec_walk(const FoldedW &W, const float (&ft)[VE], const float (&fd)[VE], int e0,
                                        float P, float E, float cbefore, float t, bool lastmode, float Z,
                                        bool *near) {
  float w[VE], pre[VE];
  vec_weights<VE>(W, ft, fd, e0, w);
  vec_prefix<VE>(w, pre);
  int pick = -1, last = -1;
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    if (w[e] > 0.f) {
      if (!lastmode && pick < 0 && __fadd_rn(P, __fadd_rn(E, __fadd_rn(cbefore, pre[e]))) > t) pick = e;
      last = e;
    }
  }
  const int sel = pick >= 0 ? pick : max(last, 0);
  float hi = __fadd_rn(P, __fadd_rn(E, cbefore)), lo = hi;
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    const float x = __fadd_rn(P, __fadd_rn(E, __fadd_rn(cbefore, pre[e])));
    if (e < sel) lo = x;
    if (e == sel) hi = x;
  }
  *near = fabsf(t - hi) <= NEAR_REL * Z || fabsf(t - lo) <= NEAR_REL * Z;
  return sel;
}

// The owner CTA's part of a cluster-wide draw: the owner thread (by the
// running masses of the block scan), its vector (by the chunk's vector
// masses in wv[]), that vector's entries re-read and walked.  Returns the
// token in thread `who` (set in every thread).
template <int DT, bool VEC>
__device__ __forceinline__ int slice_owner_draw(const unsigned char *rt, const unsigned char *rd, const FoldedW &W,
                                                const DrawSlice &ds, int V, const float *wv, float P, float t,
                                                bool lastmode, float E, float cs, float Z, DrawShared &sh, int &who,
                                                bool *near) {
  constexpr int VE = Elem<DT>::VE;
  const int tid = threadIdx.x;
  who = owner_thread(P, t, E, cs, lastmode, sh);
  if (tid != who) return -1;
  const int cper = (ds.nv + NT - 1) / NT;
  const int a0 = min(ds.nv, tid * cper), a1 = min(ds.nv, a0 + cper);
  int jv = -1, jlast = -1;
  float cpre = 0.f, cb = 0.f, cb_last = 0.f;
  for (int j = a0; j < a1; ++j) {
    const float before = cpre;
    cpre = __fadd_rn(cpre, wv[j]);
    if (wv[j] > 0.f) {
      if (!lastmode && jv < 0 && __fadd_rn(P, __fadd_rn(E, cpre)) > t) {
        jv = j;
        cb = before;
      }
      jlast = j;
      cb_last = before;
    }
  }
  if (jv < 0) {
    lastmode = true;
    jv = jlast < 0 ? a0 : jlast;
    cb = cb_last;
  }
  float ft[VE], fd[VE];
  const int e0 = ds.lo + jv * VE;
  load_vec<DT, VEC>(rt, e0, V, ft);
  if (W.mode == W_RESID)
    load_vec<DT, VEC>(rd, e0, V, fd);
  else
#pragma unroll
    for (int e = 0; e < VE; ++e) fd[e] = -INFINITY;
  return e0 + vec_walk<VE>(W, ft, fd, e0, P, E, cb, t, lastmode, Z, near);
}

// Bonus draw from p (weights 2^(z c - M c)) of one target row by one CTA,
// from the row's streaming partials: the partial of (slice s, consumer warp
// w) is the mass of a contiguous vocabulary range, so warp 0 finds the range
// holding u * Z from the partials alone (their masses kept in pm[]); one
// thread per 16-byte vector of that range weighs it, a block scan over the
// vector masses finds the owner thread, and that thread walks its vector
// from registers.  Returns the token in thread `who` (set in every thread).
template <int DT, bool VEC>
__device__ __forceinline__ int bonus_draw(const Params &p, const float4 *parts, const unsigned char *row, float M,
                                          float u, float *pm, DrawShared &sh, int &who, bool *near) {
  using El = Elem<DT>;
  constexpr int VE = El::VE;
  const int tid = threadIdx.x, lane = tid & 31;
  const float c = p.c, Mc = M * c;
  const int nparts = p.C * NCW;
  if (tid < 32) {
    constexpr int BATCH = 4;
    const int per = (nparts + 31) / 32;
    const int j0 = min(nparts, lane * per), j1 = min(nparts, j0 + per);
    float sum = 0.f;
    for (int j = j0; j < j1; j += BATCH) {
      float4 v[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) v[k] = j + k < j1 ? __ldcg(parts + j + k) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const float m = v[k].x == -INFINITY ? 0.f : __fmul_rn(v[k].y, ex2(fmaf(v[k].x, c, -Mc)));
        if (j + k < j1) pm[j + k] = m;
        sum = __fadd_rn(sum, m);
      }
    }
    float Z;
    const float excl = warp_excl_scan(sum, &Z);
    const float t = u * Z;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, sum > 0.f && __fadd_rn(excl, sum) > t);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, sum > 0.f);
    int lastmode = hit == 0;
    const int wl = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == wl) {
      float pre = 0.f, P = excl, Plast = excl;
      int own = -1, lastj = j0;
      for (int j = j0; j < j1; ++j) {
        const float before = __fadd_rn(excl, pre);
        pre = __fadd_rn(pre, pm[j]);
        if (pm[j] > 0.f) {
          if (!lastmode && own < 0 && __fadd_rn(excl, pre) > t) {
            own = j;
            P = before;
          }
          lastj = j;
          Plast = before;
        }
      }
      if (own < 0) {
        own = lastj;
        P = Plast;
        lastmode = 1;
      }
      sh.bi[4] = own;
      sh.bi[5] = lastmode;
      sh.bf[4] = P;
      sh.bf[5] = t;
      sh.zdraw = Z;
    }
  }
  __syncthreads();
  const int own = sh.bi[4];
  bool lastmode = sh.bi[5] != 0;
  const float P = sh.bf[4], t = sh.bf[5], Zd = sh.zdraw;
  // the owner range: slice sl, consumer warp w of the streaming split (its
  // start is a multiple of VE; at most NT vectors)
  const int sl = own / NCW, w = own - sl * NCW;
  const int lo_s = sl * p.slice;
  const int len_s = max(0, min(p.V, lo_s + p.slice) - lo_s);
  const int nv = (len_s + VE - 1) / VE, nvw = (nv + NCW - 1) / NCW;
  const int v0 = min(nv, w * nvw), v1 = min(nv, (w + 1) * nvw);
  FoldedW W;
  W.c = c;
  W.lt = Mc;
  W.ld = 0.f;
  W.mode = W_P;
  W.excl = -1;
  float ft[VE], fd[VE], wt[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) ft[e] = fd[e] = -INFINITY;
  float cs = 0.f;
  const int e0 = lo_s + (v0 + tid) * VE;
  if (v0 + tid < v1) {
    load_vec<DT, VEC>(row, e0, p.V, ft);
    vec_weights<VE>(W, ft, fd, e0, wt);
    cs = vec_mass<VE>(wt);
  }
  float total;
  const float E = block_exclusive_scan(cs, sh.scan, &total);
  who = owner_thread(P, t, E, cs, lastmode, sh);
  if (tid != who) return -1;
  return e0 + vec_walk<VE>(W, ft, fd, e0, P, E, 0.f, t, lastmode, Zd, near);
}

// Every CTA's mass into slot `slot` of every CTA of the cluster; after the
// cluster barrier every thread of every CTA sums them in rank order (the
// same bits everywhere).
__device__ __forceinline__ float cluster_exchange(float mass, int slot, uint32_t rank, uint32_t CD, DrawShared &sh) {
  const int tid = threadIdx.x;
  if (tid < static_cast<int>(CD)) dsmem_st_f32(dsmem_addr(&sh.xz[slot][rank], static_cast<uint32_t>(tid)), mass);
  cluster_sync();
  float Z = 0.f;
  for (uint32_t r = 0; r < CD; ++r) Z = __fadd_rn(Z, sh.xz[slot][r]);
  return Z;
}

template <int DT, bool TMA>
__global__ void __launch_bounds__(NT, 4) draw_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  // dynamic: row max [R], row sumexp [R], logits at x [2K], ok [K], u [K],
  // tokens [K], folded normalisers m c + log2 S of target and draft [K+1]
  // each, draw uniforms [K+1], then (16-byte aligned) the walk buffer
  extern __shared__ __align__(16) float dsh[];
  __shared__ DrawShared sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const uint32_t CD = cluster_size();
  const int b = blockIdx.x / CD;
  const int K = p.K;
  const int R = 2 * K + 1;
  const float c = p.c;
  float *rmax = dsh, *rsum = dsh + R, *gx = dsh + 2 * R;
  int *gok = reinterpret_cast<int *>(dsh + 2 * R + 2 * K);
  float *gu = dsh + 2 * R + 3 * K;
  int *gtok = reinterpret_cast<int *>(dsh + 2 * R + 4 * K);
  float *glt = dsh + 2 * R + 5 * K, *gld = glt + K + 1, *gw = gld + K + 1;
  float *wbuf = dsh + p.wbuf_off / 4;

  // every CTA of the cluster must be running before any DSMEM store: arrive
  // now, wait before the first store
  cluster_arrive_relaxed();
  // the next kernel on the stream may start its set-up (it waits for this
  // grid to complete before touching memory)
  pdl_launch_dependents();

  // ---- inputs (not produced by the first launch): the draft count, tokens,
  // their logits, the uniforms of the tests (slot 0) and of the draw at
  // every position (slot 1).  A point-mass draft has draft logit 0 at x and
  // draft normalisers (0, 1), so q(x) = 1.
  const int kc = p.counts ? __ldg(p.counts + b) : K;
  const bool bad_count = kc < 0 || kc > K;
  const int kb = bad_count ? 0 : kc;  // drafts of this sequence
  if (tid < 4) {
    sh.mrej[tid] = 0ull;
    sh.mnear[tid] = 0ull;
    sh.mbad[tid] = 0ull;
  }
  for (int i = tid; i < K; i += NT) {
    const int x = __ldg(p.tokens + static_cast<size_t>(b) * K + i);
    const int ok = i >= kb || (x >= 0 && x < p.V);  // drafts past the count are not read
    gtok[i] = x;
    gok[i] = ok;
    gx[2 * i] = (ok && i < kb) ? E::load(target_row<DT>(p, b, i), x) : 0.f;
    gx[2 * i + 1] = (ok && i < kb && !p.point) ? E::load(draft_row<DT>(p, b, i), x) : 0.f;
    gu[i] = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u);
  }
  for (int i = tid; i <= K; i += NT)
    gw[i] = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 1u);
  __syncthreads();  // the inputs, for the warps that take the tests below
  pdl_wait();  // the row partials of the first launch are complete and visible
  // the status word is final now (only the first launch sets its timeout
  // bit); read here, its latency hides behind the partials' loads
  const bool timed_out = stream_timed_out(p);
  if (blockIdx.x == 0 && tid < p.nshard) p.tickets[tid * TICKET_STRIDE] = 0;  // for the next call

  // ---- normalisers of all 2K+1 rows (target 0..K, draft 0..K-1), one job
  // (row pair, or the bonus row) per warp; the warp of position i < kb also
  // takes its acceptance test and records it in the sequence's bit masks
  const int nparts = p.C * NCW;
  for (int i = warp; i <= K; i += NWARP) {
    float mt, st, md, sd;
    warp_job_norms(p.partials + static_cast<size_t>(job_of(p, b, i)) * nparts, nparts, c, i < K && !p.point, mt,
                   st, md, sd);
    if (lane == 0) {
      const float mdr = p.point ? 0.f : md, sdr = p.point ? 1.f : sd;
      rmax[i] = mt;
      rsum[i] = st;
      glt[i] = __fadd_rn(__fmul_rn(mt, c), log2f(st));
      gld[i] = (i < K && !p.point) ? __fadd_rn(__fmul_rn(md, c), log2f(sd)) : 0.f;
      if (i < K) {
        rmax[K + 1 + i] = mdr;
        rsum[K + 1 + i] = sdr;
      }
      if (i < kb) {
        const int wd = i >> 6;
        const unsigned long long bit = 1ull << (i & 63);
        const float a = fmaf(gx[2 * i], c, -(mt * c));
        const float d = fmaf(gx[2 * i + 1], c, -(mdr * c));
        const float ratio = ex2(a - d) * (sdr / st);  // p_i(x_i) / q_i(x_i)
        if (!gok[i]) atomicOr(&sh.mbad[wd], bit);
        if (!(gu[i] < ratio)) atomicOr(&sh.mrej[wd], bit);
        if (isfinite(ratio) && fabsf(gu[i] - ratio) <= NEAR_REL * fmaxf(ratio, 0x1p-24f))
          atomicOr(&sh.mnear[wd], bit);
      }
    }
  }
  __syncthreads();

  // ---- n = the first reject, or kb; a draft token out of range is an
  // error; a test up to n near its boundary is counted
  int n = kb, err = bad_count;
  bool near_acc = false;
  if (kb <= 64) {  // one word (uniform in the CTA)
    const unsigned long long r = sh.mrej[0];
    if (r) n = __ffsll(static_cast<long long>(r)) - 1;
    if (sh.mbad[0]) err = 1;
    near_acc = (sh.mnear[0] & (n >= 63 ? ~0ull : (2ull << n) - 1ull)) != 0ull;
  } else {
    for (int wd = 3; wd >= 0; --wd) {
      const unsigned long long r = sh.mrej[wd];
      if (r) n = wd * 64 + __ffsll(static_cast<long long>(r)) - 1;
      if (sh.mbad[wd]) err = 1;
    }
    for (int wd = 0; wd < 4; ++wd) {  // the tests up to and including position n
      const int hi = n - wd * 64;       // highest bit of this word that counts
      const unsigned long long upto = hi >= 63 ? ~0ull : (hi < 0 ? 0ull : (2ull << hi) - 1ull);
      if (sh.mnear[wd] & upto) near_acc = true;
    }
  }
  int32_t *out = p.out_tokens + static_cast<size_t>(b) * (K + 1);
  if (rank == 0) {
    for (int r = tid; r < R; r += NT) {
      if (p.out_row_max) p.out_row_max[static_cast<size_t>(b) * R + r] = rmax[r];
      if (p.out_row_sumexp) p.out_row_sumexp[static_cast<size_t>(b) * R + r] = rsum[r];
    }
    if (err) {
      for (int e = tid; e <= K; e += NT) out[e] = -1;
      if (tid == 0) {
        p.out_n[b] = -1;
        atomicOr(p.status, ST_TOKEN);
        if (p.stats) atomicAdd(&p.stats->errors, 1ull);
      }
    }
  }
  cluster_wait();  // every peer is running (pairs with the arrive above)
  if (err) return;
  if (timed_out) {
    if (rank == 0) {
      for (int e = tid; e <= K; e += NT) out[e] = -1;
      if (tid == 0) p.out_n[b] = -1;
    }
    return;
  }

  if (n == kb) {
    // ---- bonus: rank 0 draws from p at position kb using the streaming
    // partials (the target half of a pair job's partials when kb < K)
    if (rank == 0) {
      const float u = gw[kb];
      int who;
      bool nd = false;
      const int token = bonus_draw<DT, TMA>(p, p.partials + static_cast<size_t>(job_of(p, b, kb)) * nparts,
                                            target_row<DT>(p, b, kb), rmax[kb], u, wbuf, sh, who, &nd);
      if (warp == (who >> 5)) {
        const int tk = __shfl_sync(0xFFFFFFFFu, token, who & 31);
        const bool near = __shfl_sync(0xFFFFFFFFu, static_cast<int>(nd), who & 31) || near_acc;
        for (int j = lane; j <= K; j += 32) out[j] = j < kb ? gtok[j] : (j == kb ? tk : -1);
        if (lane == 0) {
          timer_max(p, 2);
          p.out_n[b] = kb;
          if (p.stats) {
            atomicAdd(&p.stats->sequences, 1ull);
            atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(kb));
            atomicAdd(&p.stats->bonus, 1ull);
            if (near) atomicAdd(&p.stats->near_boundary, 1ull);
          }
        }
      }
    }
    return;
  }

  // ---- the residual draw at position n over the cluster
  // (point mass: the residual max(0, p - q) is p without the draft token)
  const unsigned char *rt = target_row<DT>(p, b, n);
  const unsigned char *rd = p.point ? rt : draft_row<DT>(p, b, n);
  DrawSlice ds;
  ds.set(static_cast<int>(rank), p.slice_d, p.V, VE);
  FoldedW W;
  W.c = c;
  W.lt = glt[n];
  W.ld = gld[n];
  W.mode = p.point ? W_P_EXCL : W_RESID;
  W.excl = p.point ? gtok[n] : -1;
  const float u = gw[n];
  int fallback = 0, slot = 0;
  float Ex, cs;
  float Z = cluster_exchange(slice_weigh<DT, TMA>(rt, rd, W, ds, p.V, wbuf, sh, Ex, cs), slot, rank, CD, sh);
  if (!(Z > 0.f)) {  // no residual mass in fp32: draw from p at this position
    W.mode = p.point ? W_P_EXCL : W_P;
    fallback = 1;
    slot = 1;
    Z = cluster_exchange(slice_weigh<DT, TMA>(rt, rd, W, ds, p.V, wbuf, sh, Ex, cs), slot, rank, CD, sh);
  }
  if (tid == 0) find_owner_cta(u, Z, slot, CD, sh);
  __syncthreads();
  // No DSMEM access follows the last exchange, so only the owner CTA goes on.
  if (static_cast<int>(rank) != sh.bi[2]) return;
  int who;
  bool nd = false;
  const int token = slice_owner_draw<DT, TMA>(rt, rd, W, ds, p.V, wbuf, sh.bf[0], sh.bf[1], sh.bi[3] != 0, Ex, cs,
                                              Z, sh, who, &nd);
  if (warp != (who >> 5)) return;
  const int tk = __shfl_sync(0xFFFFFFFFu, token, who & 31);
  const bool near = __shfl_sync(0xFFFFFFFFu, static_cast<int>(nd), who & 31) || near_acc;
  for (int j = lane; j <= K; j += 32) out[j] = j < n ? gtok[j] : (j == n ? tk : -1);
  if (lane == 0) {
    timer_max(p, 2);
    p.out_n[b] = n;
    if (p.stats) {
      atomicAdd(&p.stats->sequences, 1ull);
      atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(n));
      atomicAdd(&p.stats->resampled, 1ull);
      if (fallback) atomicAdd(&p.stats->residual_fallbacks, 1ull);
      if (near) atomicAdd(&p.stats->near_boundary, 1ull);
    }
  }
}

// ======================================================================
// B''. tree_draw_kernel: stochastic tree verification, one cluster per tree.
// ======================================================================
// The candidates (children) of a node are tried in index order.  With r the
// current target distribution at the node (r = p at first), candidate x is
// accepted iff u < r(x)/q(x); on a reject r becomes max(0, p - a q)/W with
// a += W and W = the mass of max(0, p - a q), weighed over the node's row
// pair by the whole cluster.  An accepted candidate becomes the current
// node; if every candidate is rejected the token is drawn from r with the
// masses of that last weighing; an accepted leaf draws a bonus token from its
// own p, from its streaming partials.  Uniforms: the test of child c uses
// (b, c - 1, slot 0), the draw at node u uses (b, u, slot 1), so that a
// chain-shaped tree is exactly the chain verification.  Every CTA of the
// cluster takes the same decisions from the same bits.
// Pages: the chain rule of blog.oscine.io "投机解码：让大模型「猜」着跑的数学魔术"
// (§"验收标准的精确数学", §"拒绝之后怎么办？——残差分布") applied sibling by
// sibling; infra-guide "5.3 Medusa, EAGLE và MTP" §9 (a tree is not lossless
// by itself) and §3 (one committed path).
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT, 4) tree_draw_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  // dynamic: parent [N], tokens [N], each node's logits at its token in its
  // parent's target and draft rows [N] + [N], acceptance uniforms [N], the
  // current node's children [N], then (16-byte aligned) the walk buffer
  extern __shared__ __align__(16) float dsh[];
  __shared__ DrawShared sh;
  __shared__ float nrm[4];  // the current node's (max, sumexp) of target and draft
  __shared__ int tst[2];    // error bits, number of children of the current node

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const uint32_t CD = cluster_size();
  const int b = blockIdx.x / CD;
  const int N = p.K;
  const float c = p.c;
  int *s_par = reinterpret_cast<int *>(dsh);
  int *s_tok = s_par + N;
  float *s_gt = reinterpret_cast<float *>(s_tok + N);
  float *s_gd = s_gt + N;
  float *s_u = s_gd + N;
  int *s_kids = reinterpret_cast<int *>(s_u + N);
  float *wbuf = dsh + p.wbuf_off / 4;

  cluster_arrive_relaxed();  // every peer must run before any DSMEM store
  pdl_launch_dependents();
  if (tid == 0) tst[0] = 0;
  __syncthreads();
  // ---- inputs: the tree, the node tokens, their logits, the uniforms
  for (int cn = tid; cn < N; cn += NT) {
    const int pu = __ldg(p.parent + static_cast<size_t>(b) * p.parent_stride + cn);
    const int x = __ldg(p.tokens + static_cast<size_t>(b) * N + cn);
    int bad = 0;
    if (cn == 0) {
      bad = pu != -1 ? 2 : 0;
    } else {
      if (pu < 0 || pu >= cn) bad |= 2;
      if (x < 0 || x >= p.V) bad |= 1;
    }
    s_par[cn] = pu;
    s_tok[cn] = x;
    s_gt[cn] = (cn > 0 && !bad) ? E::load(target_row<DT>(p, b, pu), x) : 0.f;
    s_gd[cn] = (cn > 0 && !bad) ? E::load(draft_row<DT>(p, b, pu), x) : 0.f;
    s_u[cn] = cn > 0 ? philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(cn - 1), 0u) : 0.f;
    if (bad) atomicOr(&tst[0], bad);
  }
  __syncthreads();
  if (!(tst[0] & 2)) {  // every node within max_depth of the root
    for (int cn = tid; cn < N; cn += NT) {
      int d = 0;
      for (int a = cn; a > 0 && d <= p.max_depth; a = s_par[a]) ++d;
      if (d > p.max_depth) atomicOr(&tst[0], 2);
    }
  }
  __syncthreads();
  pdl_wait();  // the row partials of the first launch are complete and visible
  // final now (only the first launch sets the timeout bit); read before the
  // cluster barrier, so its latency hides behind it
  const bool timed_out = stream_timed_out(p);
  if (blockIdx.x == 0 && tid < p.nshard) p.tickets[tid * TICKET_STRIDE] = 0;  // for the next call
  const int err = tst[0];
  const int W1 = p.max_depth + 1;
  int32_t *path = p.out_tokens + static_cast<size_t>(b) * W1;
  cluster_wait();  // pairs with the arrive above
  if (!err && timed_out) {
    if (rank == 0) {
      for (int j = tid; j < W1; j += NT) path[j] = -1;
      if (tid == 0) p.out_n[b] = -1;
    }
    return;
  }
  if (err) {
    if (rank == 0) {
      for (int j = tid; j < W1; j += NT) path[j] = -1;
      if (tid == 0) {
        p.out_n[b] = -1;
        atomicOr(p.status, (err & 2) ? ST_PARENT : ST_TOKEN);
      }
    }
    return;
  }

  const int nparts = p.C * NCW;
  DrawSlice ds;
  ds.set(static_cast<int>(rank), p.slice_d, p.V, VE);
  int node = 0, len = 0, slot = 0;
  for (;;) {
    // ---- the children of `node` in index order, and its normalisers
    if (warp == 0) {
      int cnt = 0;
      for (int base = node + 1; base < N; base += 32) {
        const int cn = base + lane;
        const bool is = cn < N && s_par[cn] == node;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, is);
        if (is) s_kids[cnt + __popc(m & ((1u << lane) - 1u))] = cn;
        cnt += __popc(m);
      }
      float mt, st, md, sd;
      warp_job_norms(p.partials + static_cast<size_t>(job_of(p, b, node)) * nparts, nparts, c, cnt > 0, mt,
                     st, md, sd);
      if (lane == 0) {
        nrm[0] = mt;
        nrm[1] = st;
        nrm[2] = md;
        nrm[3] = sd;
        tst[1] = cnt;
      }
    }
    __syncthreads();
    const int nk = tst[1];
    const float mt = nrm[0], st = nrm[1], md = nrm[2], sd = nrm[3];
    const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(node), 1u);
    if (nk == 0) {  // an accepted leaf: the bonus token from p (rank 0)
      if (rank == 0) {
        const int token = draw_p_from_partials<DT>(
            p, p.partials + static_cast<size_t>(job_of(p, b, node)) * nparts, target_row<DT>(p, b, node), mt, u,
            wbuf, sh);
        for (int j = tid; j < W1; j += NT)
          if (j >= len) path[j] = j == len ? token : -1;
        if (tid == 0) {
          p.out_n[b] = len + 1;
          timer_max(p, 2);
        }
      }
      return;
    }
    const unsigned char *rt = target_row<DT>(p, b, node), *rd = draft_row<DT>(p, b, node);
    Weights W;
    W.c = c;
    W.mtc = mt * c;
    W.mdc = md * c;
    W.inv_st = 1.f / st;
    W.resid = true;
    W.excl = -1;
    const float inv_sd = 1.f / sd;
    float a = 0.f, Wk = 1.f;
    int next = -1, vanished = 0, last_slot = 0;
    for (int k = 0; k < nk; ++k) {
      const int cn = s_kids[k];
      const float at = fmaf(s_gt[cn], c, -(mt * c));
      const float ad = fmaf(s_gd[cn], c, -(md * c));
      const float rho = ex2(at - ad) * (sd / st);  // p(x) / q(x)
      const float ratio = k == 0 ? rho : fmaxf(rho - a, 0.f) / Wk;  // r(x) / q(x)
      if (s_u[cn] < ratio) {
        next = cn;
        break;
      }
      // reject: r <- norm(max(0, r - q)) = max(0, p - a q) / W
      a = __fadd_rn(a, Wk);
      W.inv_sd = __fmul_rn(a, inv_sd);
      last_slot = slot;
      Wk = cluster_weigh<DT, TMA>(rt, rd, W, ds, slot, rank, CD, sh);
      slot ^= 1;
      if (!(Wk > 0.f)) {
        vanished = 1;
        break;
      }
    }
    if (next >= 0) {
      if (rank == 0 && tid == 0) path[len] = s_tok[next];
      ++len;
      node = next;
      __syncthreads();  // s_kids, nrm and tst are rewritten for the next node
      continue;
    }
    // ---- every candidate rejected: the draw at this node
    int token;
    if (vanished) {  // no residual mass in fp32: draw from p at this node (rank 0)
      if (rank != 0) return;
      token = draw_p_from_partials<DT>(p, p.partials + static_cast<size_t>(job_of(p, b, node)) * nparts, rt, mt,
                                       u, wbuf, sh);
    } else {
      if (tid == 0) find_owner_cta(u, Wk, last_slot, CD, sh);
      __syncthreads();
      // no DSMEM access follows the last exchange: only the owner CTA goes on
      if (static_cast<int>(rank) != sh.bi[2]) return;
      token = owner_walk<DT, TMA>(rt, rd, W, ds, wbuf, sh);
    }
    for (int j = tid; j < W1; j += NT)
      if (j >= len) path[j] = j == len ? token : -1;
    if (tid == 0) {
      p.out_n[b] = len + 1;
      timer_max(p, 2);
    }
    return;
  }
}

// ======================================================================
// B'. finish_kernel: greedy chain and greedy tree, one CTA per sequence.
// ======================================================================
__global__ void __launch_bounds__(NT) finish_kernel(const Params p) {
  extern __shared__ __align__(16) int ish[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int J = p.J;
  int *s_amax = ish;                                        // [J]
  int *s_tok = ish + J;                                     // [J]
  float *s_vmax = reinterpret_cast<float *>(ish + 2 * J);  // [J]

  const int ntok = p.kind == KIND_TREE ? J : p.K;
  int *s_par = ish + 3 * J;  // tree: parents [N]
  pdl_launch_dependents();  // the next kernel may start its set-up
  // inputs the first launch does not write: tokens (and parents)
  for (int e = tid; e < ntok; e += NT) s_tok[e] = __ldg(p.tokens + static_cast<size_t>(b) * ntok + e);
  if (p.kind == KIND_TREE)
    for (int e = tid; e < J; e += NT) s_par[e] = __ldg(p.parent + static_cast<size_t>(b) * p.parent_stride + e);
  pdl_wait();
  // final now (only the first launch sets the timeout bit); consulted after
  // the partials' folds, so its latency hides behind their loads
  const bool timed_out = stream_timed_out(p);
  if (b == 0 && tid < p.nshard) p.tickets[tid * TICKET_STRIDE] = 0;  // for the next call
  const int nparts = p.C * NCW;
  // rows of at most 4 partials per lane: a warp loads up to FIN_ROWS of its
  // rows at once (one round trip for all), then folds each in the same order
  constexpr int FIN_ROWS = 8;
  for (int r0 = warp; nparts <= 32 * 4 && r0 < J; r0 += NWARP * FIN_ROWS) {
    float4 a[FIN_ROWS][4];
#pragma unroll
    for (int q = 0; q < FIN_ROWS; ++q) {
      const int r = r0 + q * NWARP;
      const float4 *parts = p.partials + static_cast<size_t>(r < J ? job_of(p, b, r) : 0) * nparts;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = lane + 32 * k;
        a[q][k] = (r < J && j < nparts) ? __ldcg(parts + j)
                                        : make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f);
      }
    }
#pragma unroll
    for (int q = 0; q < FIN_ROWS; ++q) {
      const int r = r0 + q * NWARP;
      if (r >= J) break;  // warp-uniform
      float v = -INFINITY;
      int idx = INT_MAX;
#pragma unroll
      for (int k = 0; k < 4; ++k) am_combine(v, idx, a[q][k].x, __float_as_int(a[q][k].y));
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, off);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
        am_combine(v, idx, v2, i2);
      }
      if (lane == 0) {
        s_amax[r] = idx == INT_MAX ? 0 : idx;  // every logit -inf: first index
        s_vmax[r] = v;
      }
    }
  }
  for (int r = warp; nparts > 32 * 4 && r < J; r += NWARP) {
    float v = -INFINITY;
    int idx = INT_MAX;
    const float4 *parts = p.partials + static_cast<size_t>(job_of(p, b, r)) * nparts;
    for (int base = 0; base < nparts; base += 32 * PARTS_PER_LANE) {
      float4 a[PARTS_PER_LANE];
#pragma unroll
      for (int k = 0; k < PARTS_PER_LANE; ++k) {
        const int j = base + lane + 32 * k;
        a[k] = j < nparts ? __ldcg(parts + j) : make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < PARTS_PER_LANE; ++k) am_combine(v, idx, a[k].x, __float_as_int(a[k].y));
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, off);
      const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
      am_combine(v, idx, v2, i2);
    }
    if (lane == 0) {
      s_amax[r] = idx == INT_MAX ? 0 : idx;  // every logit -inf: first index
      s_vmax[r] = v;
    }
  }
  __syncthreads();
  if (timed_out) {  // the partials may be incomplete: no outputs drawn from them
    const int W = p.kind == KIND_TREE ? p.max_depth + 1 : p.K + 1;
    for (int e = tid; e < W; e += NT) p.out_tokens[static_cast<size_t>(b) * W + e] = -1;
    if (tid == 0) p.out_n[b] = -1;
    return;
  }

  if (p.kind == KIND_GREEDY_CHAIN) {
    const int K = p.K, R = 2 * K + 1;
    if (p.out_row_max || p.out_row_sumexp)
      for (int r = tid; r < R; r += NT) {
        if (p.out_row_max) p.out_row_max[static_cast<size_t>(b) * R + r] = r <= K ? s_vmax[r] : NAN;
        if (p.out_row_sumexp) p.out_row_sumexp[static_cast<size_t>(b) * R + r] = NAN;
      }
    if (tid == 0) {
      const int kc = p.counts ? __ldg(p.counts + b) : K;  // drafts of this sequence
      const int kb = (kc < 0 || kc > K) ? 0 : kc;
      int nacc = kb, err = kc < 0 || kc > K;
      for (int e = 0; e < kb; ++e) {
        const int x = s_tok[e];
        if (x < 0 || x >= p.V) err = 1;
        if (nacc == kb && x != s_amax[e]) nacc = e;
      }
      int32_t *out = p.out_tokens + static_cast<size_t>(b) * (K + 1);
      for (int e = 0; e <= K; ++e)
        out[e] = err ? -1 : (e < nacc ? s_tok[e] : (e == nacc ? s_amax[nacc] : -1));
      p.out_n[b] = err ? -1 : nacc;
      timer_max(p, 2);
      if (err) atomicOr(p.status, ST_TOKEN);
      if (p.stats) {
        if (err) {
          atomicAdd(&p.stats->errors, 1ull);
        } else {
          atomicAdd(&p.stats->sequences, 1ull);
          atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(nacc));
          atomicAdd(nacc == kb ? &p.stats->bonus : &p.stats->resampled, 1ull);
        }
      }
    }
    return;
  }

  // tree: J = N nodes.  Node c (c >= 1) is accepted iff every edge on its
  // path to the root is: its token equals the argmax of its parent's row.
  // Every thread takes its nodes and walks their ancestors (parent < child,
  // so a walk ends at the root within max_depth steps, else the tree is too
  // deep); the deepest accepted node, lowest index first, is the largest
  // key (depth, inverted index) of a block-wide maximum.
  const int N = J;
  __shared__ int s_bad[2];  // a malformed parent (or too deep a tree), a token out of range
  __shared__ unsigned long long s_best;
  if (tid == 0) {
    s_bad[0] = s_par[0] != -1;
    s_bad[1] = 0;
    s_best = 0ull;
  }
  __syncthreads();
  for (int c2 = 1 + tid; c2 < N; c2 += NT) {
    const int pc = s_par[c2], x = s_tok[c2];
    if (pc < 0 || pc >= c2) s_bad[0] = 1;
    if (x < 0 || x >= p.V) s_bad[1] = 1;
  }
  __syncthreads();
  if (!s_bad[0]) {
    unsigned long long best = 0ull;
    for (int c2 = tid; c2 < N; c2 += NT) {
      int d = 0;
      bool acc = true;
      for (int a = c2; a != 0 && d <= p.max_depth; ++d) {
        const int pa = s_par[a];
        acc = acc && s_tok[a] == s_amax[pa];
        a = pa;
      }
      if (d > p.max_depth) s_bad[0] = 1;
      else if (acc) best = max(best, (static_cast<unsigned long long>(d) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(c2)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (lane == 0) atomicMax(&s_best, best);
  }
  __syncthreads();
  if (tid == 0) {
    const int W = p.max_depth + 1;
    int32_t *path = p.out_tokens + static_cast<size_t>(b) * W;
    if (s_bad[0] || s_bad[1]) {
      for (int e = 0; e < W; ++e) path[e] = -1;
      p.out_n[b] = -1;
      atomicOr(p.status, s_bad[0] ? ST_PARENT : ST_TOKEN);
    } else {
      const int bestn = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(s_best));
      const int d = static_cast<int>(s_best >> 32);
      for (int e = d + 1; e < W; ++e) path[e] = -1;
      path[d] = s_amax[bestn];
      for (int n2 = bestn, e = d - 1; n2 != 0; n2 = s_par[n2], --e) path[e] = s_tok[n2];
      p.out_n[b] = d + 1;
      timer_max(p, 2);
    }
  }
}

// ======================================================================
// Self-test of the bounded waits: one thread waits, with the wait the row
// kernel uses, on an mbarrier that nothing arrives at.  The wait gives up
// after its limit (about a second), records ST_TIMEOUT and the kernel
// returns normally, so the context stays usable.
// ======================================================================
__global__ void wait_selftest_kernel(int32_t *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0)) atomicOr(status, ST_TIMEOUT);  // phase 0 never completes
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
