// Stochastic chain verification in one persistent launch: verify_kernel.
//
// Every CTA runs eight consumer warps, a producer warp and a control warp.
//
//  - The producer takes work from two global tickets.  Streaming items are
//    (job, vocabulary slice) with jobs in position-major order: the row pairs
//    (target i, draft i) of every sequence at position 0 first, then position
//    1, ..., and the bonus rows K last.  Residual tasks are (sequence,
//    slice) of sequences whose outcome is already known; a ready residual
//    task goes before the next streaming item.  The producer fills a ring of
//    shared-memory stages with TMA bulk copies (cp.async.bulk, completing an
//    mbarrier) and, once the consumers release a fill, hands its completion
//    to the control warp through a FIFO in shared memory.
//  - Consumer warp w reduces its contiguous share of each fill: the online
//    (max, sum of 2^((z - max) log2e / T)) of both rows of a streaming item,
//    or the residual mass sum max(0, p - q) of a residual task; one value per
//    warp goes to global memory.  The share of warp w of slice s is the
//    vocabulary range s * NCW + w.
//  - The control warp counts completed slices per job with GPU-scope
//    acquire-release atomics.  The warp that completes a row pair takes that
//    position's acceptance test (u < p(x)/q(x)); the test that fixes the
//    sequence's outcome (first reject n with all earlier positions accepted,
//    or every draft accepted and the bonus row complete) either draws the
//    bonus token from the row partials or publishes the sequence for its
//    residual draw.  The warp that completes the last residual slice of a
//    sequence finds the range holding u * Z from the range masses, walks
//    that range's CDF, and writes the sequence's outputs.
//
// The residual pass of a sequence runs while later positions still stream,
// on rows that were read moments before (L2-resident); only the sequences
// decided by the last rows leave work after the stream.
//
// Cross-CTA waits: only the producers' polls for residual tasks after the
// streaming items are gone; every wait is bounded (WAIT_LIMIT_NS) and sets
// ST_TIMEOUT when it runs out.  Method citations: see kernels.cuh.
#pragma once

#include "kernels.cuh"

namespace spec {

constexpr int NT_V = (NCW + 2) * 32;
constexpr int PRODUCER_WARP = NCW;
constexpr int CONTROL_WARP = NCW + 1;
constexpr int CTL_FIFO = 64;     // completion FIFO entries
constexpr int WALK_MAX = 1024;   // entries of one range: a consumer warp's share of a 16 KB tile

enum FillKind : int { FILL_NONE = -1, FILL_END = 0, FILL_ROWS = 1, FILL_RESID = 2 };

struct FillMeta {
  int kind;        // FillKind
  int n;           // elements per row in the tile
  int nrows;       // 1 or 2
  int out;         // index of the fill's first per-warp output
  int tag0, tag1;  // completion: ROWS (job q); RESID (sequence b, ready slot)
  int pad[2];
  float w[4];      // RESID: mtc, mdc, inv_st, inv_sd
};

struct ChainShared {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES];
  uint64_t cfull[CTL_FIFO], cfree[CTL_FIFO];
  FillMeta meta[MAX_STAGES];
  int4 fifo[CTL_FIFO];
  float wbuf[WALK_MAX];
};

// ------------------------------------------------------------ warp helpers
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

// (max, sumexp) of the target row (and of the draft row if `pair`) of one job
// from its C * NCW partials; lane l folds partials l, l + 32, ... in order,
// then a butterfly, so every lane holds the same bits.
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

// Inverse-CDF draw by one warp: the smallest entry v with C(v) > u * Z (else
// the last entry of positive weight), over a row split into nparts ranges of
// known mass (range j = slice j / NCW, share j % NCW of the consumer warps).
// mass(j) is the mass of range j, weight(v) the weight of entry v.  The range
// holding u * Z is found from the masses, and only its entries (at most
// WALK_MAX) are weighed, through `wbuf`.  Both levels compare the running
// sums exactly as they were formed, so a range or lane chosen by its total
// always yields an entry; where the range masses and the entry weights round
// differently (within fp32 rounding of a boundary) the last positive entry
// of the range is taken.  Returns the token in every lane, or -1 if Z <= 0.
template <int DT, class Mass, class Weight>
__device__ int warp_draw(const Params &p, int nparts, const Mass &mass, const Weight &weight, float u,
                         float *wbuf) {
  constexpr int VE = Elem<DT>::VE;
  const int lane = threadIdx.x & 31;
  constexpr int BATCH = 4;
  // 1. range masses; lane l holds a contiguous run of ranges
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
  if (!(Z > 0.f)) return -1;
  const float t = u * Z;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, sum > 0.f && __fadd_rn(excl, sum) > t);
  int lastmode = hit == 0;
  const int who = hit ? __ffs(hit) - 1 : 31 - __clz(__ballot_sync(0xFFFFFFFFu, sum > 0.f));
  int own = 0;
  float P = 0.f;
  if (lane == who) {
    float pre = 0.f, Plast = excl;
    int lastj = j0;
    own = -1;
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
  }
  own = __shfl_sync(0xFFFFFFFFu, own, who);
  P = __shfl_sync(0xFFFFFFFFu, P, who);
  lastmode = __shfl_sync(0xFFFFFFFFu, lastmode, who);
  // 2. the entries of range `own`
  const int sl = own / NCW, w = own - sl * NCW;
  const int lo_s = sl * p.slice;
  const int len_s = max(0, min(p.V, lo_s + p.slice) - lo_s);
  const int nv = (len_s + VE - 1) / VE, nvw = (nv + NCW - 1) / NCW;
  const int r0 = lo_s + min(len_s, w * nvw * VE);
  const int len = lo_s + min(len_s, (w + 1) * nvw * VE) - r0;  // <= WALK_MAX
  for (int e0 = 0; e0 < len; e0 += 32 * 8) {
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = e0 + 32 * k + lane;
      x[k] = e < len ? weight(r0 + e) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = e0 + 32 * k + lane;
      if (e < len) wbuf[e] = x[k];
    }
  }
  __syncwarp();
  const int cper = (len + 31) / 32;
  const int a0 = min(len, lane * cper), a1 = min(len, a0 + cper);
  float csum = 0.f;
  for (int e = a0; e < a1; ++e) csum = __fadd_rn(csum, wbuf[e]);
  float ctot;
  const float E0 = __fadd_rn(P, warp_excl_scan(csum, &ctot));
  int pick = -1;
  const unsigned hit2 = lastmode ? 0u : __ballot_sync(0xFFFFFFFFu, csum > 0.f && __fadd_rn(E0, csum) > t);
  if (hit2) {
    const int who2 = __ffs(hit2) - 1;
    if (lane == who2) {
      float pre = 0.f;
      for (int e = a0; e < a1; ++e) {
        const float x = wbuf[e];
        pre = __fadd_rn(pre, x);
        if (x > 0.f && __fadd_rn(E0, pre) > t) {
          pick = e;
          break;
        }
      }
    }
    pick = __shfl_sync(0xFFFFFFFFu, pick, who2);
  }
  if (pick < 0) {  // the last entry of positive weight in the range
    int lastp = -1;
    for (int e = a0; e < a1; ++e)
      if (wbuf[e] > 0.f) lastp = e;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) lastp = max(lastp, __shfl_xor_sync(0xFFFFFFFFu, lastp, off));
    pick = lastp < 0 ? 0 : lastp;
  }
  __syncwarp();  // wbuf is free again
  return r0 + pick;
}

// Draw from p = softmax(z / T) of one target row, by one warp, from the row's
// streaming partials (max m_j and sum s_j of range j): range mass
// s_j 2^((m_j - M) c), entry weight 2^((z - M) c).
template <int DT>
__device__ int warp_draw_p(const Params &p, const float4 *parts, const unsigned char *row, float M,
                           float u, float *wbuf) {
  const float c = p.c, Mc = M * c;
  auto mass = [&](int j) -> float {
    const float4 v = __ldcg(parts + j);
    return v.x == -INFINITY ? 0.f : __fmul_rn(v.y, ex2(fmaf(v.x, c, -Mc)));
  };
  auto weight = [&](int v) -> float { return ex2(fmaf(Elem<DT>::load(row, v), c, -Mc)); };
  const int tok = warp_draw<DT>(p, p.C * NCW, mass, weight, u, wbuf);
  return tok < 0 ? 0 : tok;  // no finite logit in the row (outside the contract)
}

// ------------------------------------------------------- control-warp steps
__device__ __forceinline__ void seq_stats(const Params &p, int n, int fallback) {
  if ((threadIdx.x & 31) == 0 && p.stats) {
    atomicAdd(&p.stats->sequences, 1ull);
    atomicAdd(&p.stats->accepted, static_cast<unsigned long long>(n));
    atomicAdd(n == p.K ? &p.stats->bonus : &p.stats->resampled, 1ull);
    if (fallback) atomicAdd(&p.stats->residual_fallbacks, 1ull);
  }
}

// Outputs of sequence b: drafts 0..n-1, then `token`, then -1.
__device__ __forceinline__ void emit(const Params &p, int b, int n, int token) {
  const int lane = threadIdx.x & 31, K = p.K;
  int32_t *out = p.out_tokens + static_cast<size_t>(b) * (K + 1);
  for (int j = lane; j <= K; j += 32)
    out[j] = j < n ? __ldg(p.tokens + static_cast<size_t>(b) * K + j) : (j == n ? token : -1);
  if (lane == 0) p.out_n[b] = n;
}

__device__ __forceinline__ void count_determined(const Params &p) {
  if ((threadIdx.x & 31) == 0) {
    __threadfence();
    atomicAdd(&p.ctl->determined, 1);
  }
}

// The outcome of sequence b is known: n = first rejected position, or K.
template <int DT>
__device__ void ctl_trigger(const Params &p, int b, int n, float *wbuf) {
  const int lane = threadIdx.x & 31, K = p.K;
  int bad = 0;
  for (int j = lane; j < K; j += 32) {
    const int x = __ldg(p.tokens + static_cast<size_t>(b) * K + j);
    bad |= x < 0 || x >= p.V;
  }
  if (__any_sync(0xFFFFFFFFu, bad)) {  // a draft token outside [0, V): the sequence is an error
    int32_t *out = p.out_tokens + static_cast<size_t>(b) * (K + 1);
    for (int j = lane; j <= K; j += 32) out[j] = -1;
    if (lane == 0) {
      p.out_n[b] = -1;
      atomicOr(p.status, ST_TOKEN);
      if (p.stats) atomicAdd(&p.stats->errors, 1ull);
    }
    count_determined(p);
    return;
  }
  __threadfence();
  if (n == K) {  // every draft accepted: the bonus token from p_K
    const float M = __ldcg(&p.norms[static_cast<size_t>(b) * (K + 1) + K].x);
    const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(K), 1u);
    const float4 *parts = p.partials + static_cast<size_t>(K * p.B + b) * p.C * NCW;
    const int tok = warp_draw_p<DT>(p, parts, target_row<DT>(p, b, K), M, u, wbuf);
    emit(p, b, K, tok);
    seq_stats(p, K, 0);
    count_determined(p);
    return;
  }
  // a reject at n: publish the sequence for its residual draw
  if (lane == 0) {
    const float4 nn = __ldcg(&p.norms[static_cast<size_t>(b) * (K + 1) + n]);
    ReadyRec r;
    r.b = b;
    r.n = n;
    r.mtc = nn.x * p.c;
    r.mdc = nn.z * p.c;
    r.inv_st = 1.f / nn.y;
    r.inv_sd = 1.f / nn.w;
    r.pad[0] = r.pad[1] = 0;
    const int slot = atomicAdd(&p.ctl->ready_tail, 1);
    p.ready[slot] = r;
    __threadfence();
    st_relaxed(&p.ready_flag[slot], b + 1);
  }
  count_determined(p);
}

// Outcome of sequence b from its decision bits, or -1 while unknown: the
// first rejected position r (or K) once positions 0..r are all decided.
__device__ __forceinline__ int mask_outcome(unsigned long long m, int K) {
  const unsigned dec = static_cast<unsigned>(m), rej = static_cast<unsigned>(m >> 32);
  const int r = rej ? __ffs(rej) - 1 : K;
  const unsigned need = (2u << r) - 1u;  // bits 0..r (r <= 31; 2 << 31 wraps to 0)
  return (dec & need) == need ? r : -1;
}

// Records the verdict of position i of sequence b (1 = accepted or bonus row
// complete, 2 = rejected) after its norms are written; the record that fixes
// the outcome triggers the sequence.
template <int DT>
__device__ void ctl_publish(const Params &p, int b, int i, int verdict, float *wbuf) {
  const int lane = threadIdx.x & 31, K = p.K;
  int n = -1;
  if (K <= 31) {
    if (lane == 0) {
      const unsigned long long add = (1ull << i) | (verdict == 2 ? 1ull << (32 + i) : 0ull);
      const unsigned long long old = atom_or_acq_rel(&p.seq_mask[b], add);
      const unsigned long long now = old | add;
      if (mask_outcome(old, K) < 0) n = mask_outcome(now, K);
      const unsigned all = (2u << K) - 1u;
      if ((static_cast<unsigned>(now) & all) == all) p.seq_mask[b] = 0ull;  // every position known
    }
    n = __shfl_sync(0xFFFFFFFFu, n, 0);
  } else {
    // long chains: the last of the K+1 records decides
    int last = 0;
    if (lane == 0) {
      p.pos_state[static_cast<size_t>(b) * (K + 1) + i] = verdict;
      last = atom_add_acq_rel(&p.dec_count[b], 1) == K;
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      __syncwarp();
      __threadfence();
      int first = K;
      for (int j = lane; j < K; j += 32)
        if (__ldcg(&p.pos_state[static_cast<size_t>(b) * (K + 1) + j]) == 2) {
          first = j;
          break;
        }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, off));
      n = first;
      __syncwarp();
      for (int j = lane; j <= K; j += 32) p.pos_state[static_cast<size_t>(b) * (K + 1) + j] = 0;
      if (lane == 0) p.dec_count[b] = 0;
    }
  }
  if (n >= 0) ctl_trigger<DT>(p, b, n, wbuf);
}

// Every slice of row pair i of sequence b is reduced: the acceptance test.
template <int DT>
__device__ void ctl_decide(const Params &p, int b, int i, float *wbuf) {
  const int lane = threadIdx.x & 31, K = p.K;
  const float c = p.c;
  // the draft token and its two logits, in flight with the partial loads
  float gt = 0.f, gd = 0.f;
  int ok = 0;
  if (lane == 0) {
    const int x = __ldg(p.tokens + static_cast<size_t>(b) * K + i);
    ok = x >= 0 && x < p.V;
    if (ok) {
      gt = Elem<DT>::load(target_row<DT>(p, b, i), x);
      gd = Elem<DT>::load(draft_row<DT>(p, b, i), x);
    }
  }
  float mt, st, md, sd;
  const int q = i * p.B + b;
  warp_norms(p.partials + static_cast<size_t>(q) * p.C * NCW, p.C * NCW, c, true, mt, st, md, sd);
  int verdict = 0;
  if (lane == 0) {
    const float a = fmaf(gt, c, -(mt * c));
    const float d = fmaf(gd, c, -(md * c));
    const float ratio = ex2(a - d) * (sd / st);  // p_i(x_i) / q_i(x_i)
    const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u);
    verdict = (ok && u < ratio) ? 1 : 2;
    p.norms[static_cast<size_t>(b) * (K + 1) + i] = make_float4(mt, st, md, sd);
    const size_t R = 2 * static_cast<size_t>(K) + 1;
    if (p.out_row_max) {
      p.out_row_max[b * R + i] = mt;
      p.out_row_max[b * R + K + 1 + i] = md;
    }
    if (p.out_row_sumexp) {
      p.out_row_sumexp[b * R + i] = st;
      p.out_row_sumexp[b * R + K + 1 + i] = sd;
    }
  }
  ctl_publish<DT>(p, b, i, verdict, wbuf);
}

// Every slice of the bonus row of sequence b is reduced.
template <int DT>
__device__ void ctl_bonus_row(const Params &p, int b, float *wbuf) {
  const int lane = threadIdx.x & 31, K = p.K;
  float mt, st, md, sd;
  const int q = K * p.B + b;
  warp_norms(p.partials + static_cast<size_t>(q) * p.C * NCW, p.C * NCW, p.c, false, mt, st, md, sd);
  if (lane == 0) {
    p.norms[static_cast<size_t>(b) * (K + 1) + K] = make_float4(mt, st, -INFINITY, 0.f);
    const size_t R = 2 * static_cast<size_t>(K) + 1;
    if (p.out_row_max) p.out_row_max[b * R + K] = mt;
    if (p.out_row_sumexp) p.out_row_sumexp[b * R + K] = st;
  }
  ctl_publish<DT>(p, b, K, 1, wbuf);
}

// Every residual slice of sequence b is reduced: the residual draw.
template <int DT>
__device__ void ctl_residual_final(const Params &p, int b, int slot, float *wbuf) {
  const int lane = threadIdx.x & 31, K = p.K;
  const int4 *rp = reinterpret_cast<const int4 *>(p.ready + slot);
  const int4 h0 = __ldcg(rp), h1 = __ldcg(rp + 1);
  const int n = h0.y;
  Weights W;
  W.c = p.c;
  W.mtc = __int_as_float(h0.z);
  W.mdc = __int_as_float(h0.w);
  W.inv_st = __int_as_float(h1.x);
  W.inv_sd = __int_as_float(h1.y);
  W.resid = true;
  const float u = philox_uniform(p.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(n), 1u);
  const float *masses = p.rmass + static_cast<size_t>(b) * p.C * NCW;
  const unsigned char *rt = target_row<DT>(p, b, n), *rd = draft_row<DT>(p, b, n);
  auto mass = [&](int j) -> float { return __ldcg(masses + j); };
  auto weight = [&](int v) -> float { return W(Elem<DT>::load(rt, v), Elem<DT>::load(rd, v)); };
  int tok = warp_draw<DT>(p, p.C * NCW, mass, weight, u, wbuf);
  int fallback = 0;
  if (tok < 0) {  // no residual mass in fp32 (p_n == q_n): draw from p_n
    fallback = 1;
    const float M = __ldcg(&p.norms[static_cast<size_t>(b) * (K + 1) + n].x);
    tok = warp_draw_p<DT>(p, p.partials + static_cast<size_t>(n * p.B + b) * p.C * NCW, rt, M, u, wbuf);
  }
  emit(p, b, n, tok);
  seq_stats(p, n, fallback);
  if (lane == 0) p.ready_flag[slot] = 0;  // every task of this slot is done
}

// ======================================================================
// verify_kernel
// ======================================================================
template <int DT, bool TMA>
__global__ void __launch_bounds__(NT_V, 2) verify_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VE = E::VE;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ ChainShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, C = p.C, B = p.B, K = p.K;
  const int nparts = C * NCW;
  const float c = p.c;
  const size_t row_bytes = static_cast<size_t>(p.tile) * E::BYTES;
  auto stage_row = [&](int s, int r) -> unsigned char * {
    return dyn + (static_cast<size_t>(s) * 2 + r) * row_bytes;
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], NCW);
    }
    for (int f = 0; f < CTL_FIFO; ++f) {
      mbar_init(&sh.cfull[f], 1);
      mbar_init(&sh.cfree[f], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  bool tmo = false;
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    const int nitems = p.njobs * C;
    int pseq = 0, pdone = 0, cseq = 0;  // fills issued, fills handed in, FIFO entries
    // Only lane 0 waits on the producer's barriers and only lane 0 arrives on
    // them; the warp learns the outcome through the shuffle.  (Were every
    // lane to wait, a lane that polls after lane 0 has already acted could
    // find the next phase complete and wait for a parity that never returns.)
    auto wait0 = [&](uint64_t *bar, uint32_t parity) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(bar, parity);
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) tmo = true;
    };
    auto ctl_push = [&](int kind, int t0, int t1) {
      const int f = cseq % CTL_FIFO;
      wait0(&sh.cfree[f], ((cseq / CTL_FIFO) & 1) ^ 1);
      if (lane == 0) {
        sh.fifo[f] = make_int4(kind, t0, t1, 0);
        mbar_arrive(&sh.cfull[f]);
      }
      __syncwarp();
      ++cseq;
    };
    auto observe = [&]() {  // the oldest fill in flight is released: hand it in
      const int s = pdone % S;
      wait0(&sh.empty[s], (pdone / S) & 1);
      ctl_push(sh.meta[s].kind, sh.meta[s].tag0, sh.meta[s].tag1);
      ++pdone;
    };
    auto acquire = [&]() -> int {
      while (pseq - pdone >= S && !tmo) observe();
      return pseq % S;
    };
    auto issue = [&](int s, const unsigned char *rt, const unsigned char *rd, int n, int nrows) {
      if (TMA) {
        if (lane == 0) {
          const uint32_t bytes = static_cast<uint32_t>(n) * E::BYTES;
          mbar_arrive_expect_tx(&sh.full[s], bytes * nrows);
          bulk_g2s(stage_row(s, 0), rt, bytes, &sh.full[s]);
          if (nrows == 2) bulk_g2s(stage_row(s, 1), rd, bytes, &sh.full[s]);
        }
      } else {
        const int npad = (n + VE - 1) / VE * VE;
        for (int r = 0; r < nrows; ++r) {
          const unsigned char *g = r ? rd : rt;
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
        if (lane == 0) mbar_arrive(&sh.full[s]);
      }
      ++pseq;
    };

    // lane 0 holds the tickets: the next streaming item and one residual task
    // (task index held = slot * C + slice).  Streaming items come from this
    // CTA's shard first, then from the others once it is used up; residual
    // tickets always from this CTA's shard.
    const int ns = p.nshard;
    const int rshard = static_cast<int>(blockIdx.x) % ns;
    int ishard = rshard, iempty = 0;
    auto take_item = [&]() -> int {
      while (iempty < ns) {
        const long long it =
            static_cast<long long>(atomicAdd(&p.ctl->item[ishard * SHARD_STRIDE], 1)) * ns + ishard;
        if (it < nitems) return static_cast<int>(it);
        ++iempty;
        ishard = ishard + 1 == ns ? 0 : ishard + 1;
      }
      return nitems;
    };
    auto take_task = [&]() -> int {
      return atomicAdd(&p.ctl->res[rshard * SHARD_STRIDE], 1) * ns + rshard;
    };
    int item = 0, held = 0, flag = 0;
    if (lane == 0) {
      item = take_item();
      held = take_task();
    }
    bool finished = false;
    while (!finished && !tmo) {
      const int s = acquire();
      if (tmo) break;
      int act = 0;
      if (lane == 0) act = flag ? 1 : (item < nitems ? 2 : 0);
      act = __shfl_sync(0xFFFFFFFFu, act, 0);
      if (act == 1) {
        // -------- a residual task: slice (held mod C) of a published sequence
        int4 h0 = make_int4(0, 0, 0, 0), h1 = h0;
        int tk = 0;
        if (lane == 0) {
          tk = held;
          __threadfence();
          const int4 *rp = reinterpret_cast<const int4 *>(p.ready + held / C);
          h0 = __ldcg(rp);
          h1 = __ldcg(rp + 1);
        }
        tk = __shfl_sync(0xFFFFFFFFu, tk, 0);
        const int b = __shfl_sync(0xFFFFFFFFu, h0.x, 0), n = __shfl_sync(0xFFFFFFFFu, h0.y, 0);
        const int slot = tk / C, sl = tk - slot * C;
        const int lo = sl * p.slice, len = max(0, min(p.V, lo + p.slice) - lo);
        if (len == 0) {
          if (lane < NCW) p.rmass[static_cast<size_t>(b) * nparts + sl * NCW + lane] = 0.f;
          __syncwarp();
          ctl_push(FILL_RESID, b, slot);
        } else {
          if (lane == 0) {
            FillMeta m;
            m.kind = FILL_RESID;
            m.n = len;
            m.nrows = 2;
            m.out = b * nparts + sl * NCW;
            m.tag0 = b;
            m.tag1 = slot;
            m.pad[0] = m.pad[1] = 0;
            m.w[0] = __int_as_float(h0.z);
            m.w[1] = __int_as_float(h0.w);
            m.w[2] = __int_as_float(h1.x);
            m.w[3] = __int_as_float(h1.y);
            sh.meta[s] = m;
          }
          const size_t off = static_cast<size_t>(lo) * E::BYTES;
          issue(s, target_row<DT>(p, b, n) + off, draft_row<DT>(p, b, n) + off, len, 2);
        }
        if (lane == 0) {
          held = take_task();
          flag = 0;  // polled after the next fill, once the new ticket is in
        }
        continue;
      }
      if (act == 2) {
        // -------- a streaming item: slice sl of job q = i * B + b
        const int it = __shfl_sync(0xFFFFFFFFu, item, 0);
        if (lane == 0) item = take_item();
        const int q = it / C, sl = it - q * C;
        const int i = q / B, b = q - i * B;
        const int lo = sl * p.slice, len = max(0, min(p.V, lo + p.slice) - lo);
        const int nrows = i < K ? 2 : 1;
        if (len == 0) {
          if (lane < NCW)
            p.partials[static_cast<size_t>(it) * NCW + lane] = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
          __syncwarp();
          ctl_push(FILL_ROWS, q, 0);
        } else {
          if (lane == 0) {
            FillMeta m;
            m.kind = FILL_ROWS;
            m.n = len;
            m.nrows = nrows;
            m.out = it * NCW;
            m.tag0 = q;
            m.tag1 = 0;
            m.pad[0] = m.pad[1] = 0;
            m.w[0] = m.w[1] = m.w[2] = m.w[3] = 0.f;
            sh.meta[s] = m;
          }
          const size_t off = static_cast<size_t>(lo) * E::BYTES;
          issue(s, target_row<DT>(p, b, i) + off, nrows == 2 ? draft_row<DT>(p, b, i) + off : nullptr, len,
                nrows);
        }
        // readiness of the held residual ticket, read while the next stage frees up
        if (lane == 0) {
          const int slot = held / C;
          flag = slot < B ? ld_relaxed(&p.ready_flag[slot]) : 0;
        }
        continue;
      }
      // -------- nothing left to stream: hand in the fills in flight, then
      // wait for the held residual task or for the end of the call
      while (pdone < pseq && !tmo) observe();
      const uint64_t t0 = clock_ns();
      for (int polls = 0;; ++polls) {
        int st = 0;
        if (lane == 0) {
          const int slot = held / C;
          if (slot < B && ld_relaxed(&p.ready_flag[slot]) != 0) {
            st = 1;
          } else if (ld_relaxed(&p.ctl->determined) >= B) {
            __threadfence();  // every publication is visible: ready_tail is final
            if (slot >= ld_relaxed(&p.ctl->ready_tail)) st = 2;
          }
        }
        st = __shfl_sync(0xFFFFFFFFu, st, 0);
        if (st == 1) {
          if (lane == 0) flag = 1;
          break;
        }
        if (st == 2) {
          finished = true;
          break;
        }
        if (clock_ns() - t0 > WAIT_LIMIT_NS || polls > (1 << 22)) {
          tmo = true;
          break;
        }
        __nanosleep(256);
      }
    }
    if (!tmo) {  // end of stream: consumers, then the control warp
      const int s = acquire();
      if (!tmo) {
        if (lane == 0) {
          sh.meta[s].kind = FILL_END;
          mbar_arrive(&sh.full[s]);
        }
        __syncwarp();
        ctl_push(FILL_END, 0, 0);
      }
    }
  } else if (warp == CONTROL_WARP) {
    // ------------------------------------------------------------ control
    int k = 0;
    bool done = false;
    while (!done) {
      // every lane waits (acquiring the entry); the outcome is decided warp-wide
      const bool ok = mbar_wait_bounded(&sh.cfull[k % CTL_FIFO], (k / CTL_FIFO) & 1);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        tmo = true;
        break;
      }
      // entries k, k+1, ... that are already there, one per lane
      const int g = (k + lane) % CTL_FIFO;
      const bool rdy = lane == 0 || mbar_test(&sh.cfull[g], ((k + lane) / CTL_FIFO) & 1);
      const unsigned notrdy = ~__ballot_sync(0xFFFFFFFFu, rdy);
      const int navail = notrdy ? __ffs(notrdy) - 1 : 32;
      int4 e = make_int4(FILL_NONE, 0, 0, 0);
      if (lane < navail) {
        e = sh.fifo[g];
        mbar_arrive(&sh.cfree[g]);
      }
      k += navail;
      int last = 0;
      if (e.x == FILL_ROWS || e.x == FILL_RESID) {
        int *ctr = e.x == FILL_ROWS ? p.job_done + e.y : p.res_done + e.y;
        last = atom_add_acq_rel(ctr, 1) == C - 1;
        if (last) *ctr = 0;  // no other use of this counter in the call
      }
      done = __any_sync(0xFFFFFFFFu, e.x == FILL_END);
      unsigned lm = __ballot_sync(0xFFFFFFFFu, last);
      __syncwarp();
      while (lm) {
        const int j = __ffs(lm) - 1;
        lm &= lm - 1;
        const int kind = __shfl_sync(0xFFFFFFFFu, e.x, j);
        const int t0 = __shfl_sync(0xFFFFFFFFu, e.y, j), t1 = __shfl_sync(0xFFFFFFFFu, e.z, j);
        __threadfence();
        if (kind == FILL_ROWS) {
          const int i = t0 / B, b = t0 - i * B;
          if (i < K)
            ctl_decide<DT>(p, b, i, sh.wbuf);
          else
            ctl_bonus_row<DT>(p, b, sh.wbuf);
        } else {
          ctl_residual_final<DT>(p, t0, t1, sh.wbuf);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    Online ot, od;
    ot.init();
    od.init();
    for (int seq = 0;; ++seq) {
      const int s = seq % S;
      // every lane waits (the TMA writes become visible to it); a timeout ends
      // the loop for the whole warp
      const bool ok = mbar_wait_bounded(&sh.full[s], (seq / S) & 1);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        tmo = true;
        break;
      }
      const int kind = sh.meta[s].kind;
      if (kind == FILL_END) break;
      const int n = sh.meta[s].n, out = sh.meta[s].out;
      const int nv = (n + VE - 1) / VE;
      const int nvw = (nv + NCW - 1) / NCW;
      const int j0 = warp * nvw + lane, j1 = min(nv, (warp + 1) * nvw);
      const unsigned char *bt = stage_row(s, 0), *bd = stage_row(s, 1);
      if (kind == FILL_ROWS) {
        const int nrows = sh.meta[s].nrows;
        if (nrows == 2) {
          for (int j = j0; j < j1; j += 32) {
            const uint4 wt = lds128(bt + j * 16), wd = lds128(bd + j * 16);
            online_vec16<DT>(wt, c, ot);
            online_vec16<DT>(wd, c, od);
          }
        } else {
          for (int j = j0; j < j1; j += 32) online_vec16<DT>(lds128(bt + j * 16), c, ot);
        }
        float m_t = ot.m, s_t = ot.sum(), m_d = od.m, s_d = od.sum();
        warp_ms(m_t, s_t, c);
        if (nrows == 2) warp_ms(m_d, s_d, c);
        if (lane == 0) p.partials[static_cast<size_t>(out) + warp] = make_float4(m_t, s_t, m_d, s_d);
        ot.init();
        od.init();
      } else {
        Weights W;
        W.c = c;
        W.mtc = sh.meta[s].w[0];
        W.mdc = sh.meta[s].w[1];
        W.inv_st = sh.meta[s].w[2];
        W.inv_sd = sh.meta[s].w[3];
        W.resid = true;
        float acc = 0.f;
        for (int j = j0; j < j1; j += 32) {
          float ft[VE], fd[VE];
          E::unpack(lds128(bt + j * 16), ft);
          E::unpack(lds128(bd + j * 16), fd);
#pragma unroll
          for (int e = 0; e < VE; ++e) acc = __fadd_rn(acc, W(ft[e], fd[e]));
        }
        acc = warp_sum(acc);
        if (lane == 0) p.rmass[static_cast<size_t>(out) + warp] = acc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);  // releases the stage and orders the write above
    }
  }
  if (tmo) atomicOr(p.status, ST_TIMEOUT);
  __syncthreads();
  if (tid == 0) {  // the last CTA to finish puts the call's tickets back to zero
    __threadfence();
    if (atomicAdd(&p.ctl->exited, 1) == static_cast<int>(gridDim.x) - 1) {
      __threadfence();
      for (int k = 0; k < p.nshard; ++k) {
        p.ctl->item[k * SHARD_STRIDE] = 0;
        p.ctl->res[k * SHARD_STRIDE] = 0;
      }
      p.ctl->ready_tail = 0;
      p.ctl->determined = 0;
      p.ctl->exited = 0;
    }
  }
}

}  // namespace spec
