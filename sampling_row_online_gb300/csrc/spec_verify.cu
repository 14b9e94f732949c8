// Host side of libspec_verify.so: argument validation, launch geometry
// (cluster size, slices, tiles, stages), per-stream workspaces and the C ABI
// declared in include/spec_verify.h.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.cuh"
#include "eagle2.cuh"
#include "ngram.cuh"
#include "spec_verify.h"

namespace spec {
namespace {

thread_local std::string g_last_error;

void noalloc_forget();  // spec_verify_noalloc's cached device addresses (defined with it)

// Fault injection for tests (spec_debug_fail_launch): the n-th launch from
// now reports cudaErrorLaunchFailure without launching.  0: off.
std::atomic<int> g_fail_launch{0};

cudaError_t launch_kernel(const cudaLaunchConfig_t *cfg, const void *fn, void **args) {
  int n = g_fail_launch.load();
  while (n > 0 && !g_fail_launch.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 1) return cudaErrorLaunchFailure;  // this launch is the injected failure
  return cudaLaunchKernelExC(cfg, fn, args);
}

// An NVTX range around each entry point (free when no tool is attached), so
// that profilers can attribute kernels to calls.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

int fail(int code, const std::string &msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return SPEC_ERR_CUDA;
}

// Status word (one 256-byte slot) followed by the item tickets.
constexpr size_t CONTROL_BYTES = 256 + sizeof(int) * NSHARD * TICKET_STRIDE;
inline int *tickets_of(int32_t *status) {
  return reinterpret_cast<int *>(reinterpret_cast<unsigned char *>(status) + 256);
}

// ------------------------------------------------------------ workspaces
// Per (device, stream): the status word (never reallocated), the row
// partials of the current call (float4 per job and slice, grow-only), and a
// staging area for the host-buffer entry point.
struct Workspace {
  int device = -1;
  cudaStream_t stream = nullptr;
  int32_t *status = nullptr;  // status word, then the item tickets (zeroed once)
  float4 *partials = nullptr;
  size_t cap_parts = 0;
  unsigned char *stage = nullptr;
  size_t stage_cap = 0;
  int *ngram_done = nullptr;  // n-gram drafter: finished-CTA counters, zero between calls
  size_t ngram_cap = 0;
};

std::mutex g_mu;
std::vector<Workspace *> g_ws;

Workspace *find_ws(int device, cudaStream_t stream, bool create) {
  for (Workspace *w : g_ws)
    if (w->device == device && w->stream == stream) return w;
  if (!create) return nullptr;
  Workspace *w = new Workspace;
  w->device = device;
  w->stream = stream;
  g_ws.push_back(w);
  return w;
}

int get_ws(cudaStream_t stream, size_t nparts, Workspace **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace *w = find_ws(dev, stream, true);
  if (!w->status) {
    e = cudaMalloc(&w->status, CONTROL_BYTES);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
    e = cudaMemsetAsync(w->status, 0, CONTROL_BYTES, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  }
  if (w->cap_parts < nparts) {
    if (w->partials) {
      e = cudaFree(w->partials);  // synchronises the device: no call still uses it
      w->partials = nullptr;
      w->cap_parts = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree(partials)");
    }
    e = cudaMalloc(&w->partials, sizeof(float4) * nparts);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(partials)");
    w->cap_parts = nparts;
  }
  *out = w;
  return SPEC_OK;
}

// ------------------------------------------------------------ geometry
constexpr int DEFAULT_STAGES = 2;               // tile ring depth
constexpr int TILE_MAX_BYTES = 16 * 1024;       // tile width per row
constexpr int DRAW_SLICE_BYTES = 32 * 1024;     // draw: bytes of each row per CTA (one wave)
constexpr int DRAW_MAX_VECTORS = 16384;         // chain draw: vectors per CTA slice (64 KB of masses)
constexpr int DRAW_SLICE_BYTES_TREE = 16 * 1024;  // the same for a stochastic tree, whose draw weighs
                                                  // one row pair per rejected candidate, in sequence
constexpr int DRAW_CTAS_PER_SM = 4;             // draw: resident CTAs per SM (its launch bound)

int env_int(const char *name, int dflt, int lo, int hi) {
  const char *v = std::getenv(name);
  if (!v || !*v) return dflt;
  const int x = std::atoi(v);
  return (x >= lo && x <= hi) ? x : dflt;
}

struct KernelCache {
  const void *fn;
  int device;
  int smem_set;   // largest dynamic smem attribute set so far
  int q_smem, q_C;  // last occupancy query
  int q_result;
};
std::vector<KernelCache> g_kc;

// Dynamic-smem attribute once per (kernel, device) and size, then either the
// resident blocks per SM (C == -1: row kernel blocks, C == 0: NT-thread
// blocks) or the resident clusters of size C.
int occupancy(const void *fn, int smem, int C, int *result) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  KernelCache *kc = nullptr;
  for (auto &k : g_kc)
    if (k.fn == fn && k.device == dev) kc = &k;
  if (!kc) {
    KernelCache k{};
    k.fn = fn;
    k.device = dev;
    k.smem_set = -1;
    k.q_smem = -1;
    g_kc.push_back(k);
    kc = &g_kc.back();
    if (C > 0) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
    }
  }
  if (smem > kc->smem_set) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    kc->smem_set = smem;
    kc->q_smem = -1;
  }
  if (kc->q_smem != smem || kc->q_C != C) {
    int n = 0;
    if (C <= 0) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, C == -1 ? NT_ROW : NT, smem);
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(C, 1, 1);
      cfg.blockDim = dim3(NT, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = C;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    kc->q_smem = smem;
    kc->q_C = C;
    kc->q_result = n;
  }
  *result = kc->q_result;
  return SPEC_OK;
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 1;
  }
  return sms[dev];
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <bool ARGMAX>
const void *pick_row_kernel(int dtype, bool tma) {
  if (dtype == SPEC_F32)
    return tma ? reinterpret_cast<const void *>(&row_kernel<0, true, ARGMAX>)
               : reinterpret_cast<const void *>(&row_kernel<0, false, ARGMAX>);
  return tma ? reinterpret_cast<const void *>(&row_kernel<1, true, ARGMAX>)
             : reinterpret_cast<const void *>(&row_kernel<1, false, ARGMAX>);
}

const void *pick_tree_draw_kernel(int dtype, bool tma) {
  if (dtype == SPEC_F32)
    return tma ? reinterpret_cast<const void *>(&tree_draw_kernel<0, true>)
               : reinterpret_cast<const void *>(&tree_draw_kernel<0, false>);
  return tma ? reinterpret_cast<const void *>(&tree_draw_kernel<1, true>)
             : reinterpret_cast<const void *>(&tree_draw_kernel<1, false>);
}

const void *pick_draw_kernel(int dtype, bool tma) {
  if (dtype == SPEC_F32)
    return tma ? reinterpret_cast<const void *>(&draw_kernel<0, true>)
               : reinterpret_cast<const void *>(&draw_kernel<0, false>);
  return tma ? reinterpret_cast<const void *>(&draw_kernel<1, true>)
             : reinterpret_cast<const void *>(&draw_kernel<1, false>);
}

// Launch geometry of one call.
struct Geometry {
  const void *fa, *fb;   // row kernel, decision kernel
  int C, slice, tile, stages;
  int CD, slice_d, wbuf_off;
  int smem_a, smem_b, grid_a, nshard;
  long long nitems;
};

int plan(Params &p, int dtype, bool tma, Geometry *g) {
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const int VE = 16 / esz;
  const bool argmax = p.kind == KIND_GREEDY_CHAIN || p.kind == KIND_TREE;
  const int srows = argmax ? 1 : 2;
  const long long row_bytes = static_cast<long long>(p.V) * esz;
  // streaming items are single tiles of at most 16 KB per row
  const int C_min = static_cast<int>(std::max<long long>(1, (row_bytes + TILE_MAX_BYTES - 1) / TILE_MAX_BYTES));
  g->C = C_min;
  g->stages = DEFAULT_STAGES;
  g->fa = argmax ? pick_row_kernel<true>(dtype, tma) : pick_row_kernel<false>(dtype, tma);
  g->fb = argmax ? reinterpret_cast<const void *>(&finish_kernel)
                 : (p.kind == KIND_TREE_SAMPLE ? pick_tree_draw_kernel(dtype, tma) : pick_draw_kernel(dtype, tma));
  const int per = (p.V + g->C - 1) / g->C;
  g->slice = (per + VE - 1) / VE * VE;
  g->tile = std::min(TILE_MAX_BYTES / esz, g->slice);
  g->smem_a = g->stages * srows * g->tile * esz;
  g->nitems = static_cast<long long>(p.njobs) * g->C;
  if (g->nitems * NCW > INT_MAX) return fail(SPEC_ERR_ARG, "too many rows");
  int st, per_sm = 0;
  if ((st = occupancy(g->fa, g->smem_a, -1, &per_sm))) return st;
  if (per_sm < 1) return fail(SPEC_ERR_UNSUPPORTED, "row kernel does not fit on an SM");
  g->grid_a = static_cast<int>(std::min<long long>(g->nitems, static_cast<long long>(per_sm) * num_sms()));
  // ticket shards: a divisor of the grid (every shard the same number of
  // CTAs), at most NSHARD; a large grid with no divisor in [8, NSHARD] is
  // trimmed to a multiple of 8
  g->nshard = 1;
  for (int d = std::min(NSHARD, g->grid_a); d >= 1; --d)
    if (g->grid_a % d == 0) {
      g->nshard = d;
      break;
    }
  if (g->nshard < 8 && g->grid_a >= 64) {
    g->grid_a = g->grid_a / 8 * 8;
    g->nshard = 8;
  }
  g->CD = 1;
  g->slice_d = 0;
  g->wbuf_off = 0;
  if (argmax) {
    g->smem_b = 4 * (3 * p.J) + (p.kind == KIND_TREE ? 9 * p.J : 0) + 16;
    return SPEC_OK;
  }
  // the draw: clusters of CD CTAs, about 32 KB of each row per CTA; the walk
  // buffer holds one warp range of a CTA slice or of a streaming tile
  // chain: normalisers, logits at x, uniforms, tokens, folded normalisers,
  // draw uniforms; tree: parent, tokens,
  // logits at each token, uniforms, children of the current node
  const int base = p.kind == KIND_TREE_SAMPLE ? (4 * 6 * p.K + 15) / 16 * 16
                                              : (4 * (12 * p.K + 5) + 15) / 16 * 16;
  // CTAs per sequence: slices of DRAW_SLICE_BYTES of each row (a stochastic
  // tree's draw, a chain of weighings, takes more and narrower ones), but no more
  // CTAs than one wave of the batch holds (a grid of many waves pays each
  // CTA's fixed steps -- dependency wait, normalisers, decisions, exchange --
  // once per CTA), and at least enough that a slice stays within what its
  // walk holds: the vector masses of a chain draw's slice in the walk buffer
  // (DRAW_MAX_VECTORS), a stochastic tree's warp ranges within NT * NT entries
  const bool chain = p.kind == KIND_SAMPLE;
  const long long slice_bytes = chain ? DRAW_SLICE_BYTES : DRAW_SLICE_BYTES_TREE;
  const long long cd_size = std::max<long long>(1, (row_bytes + slice_bytes - 1) / slice_bytes);
  const long long cd_wave = std::max<long long>(1, (static_cast<long long>(DRAW_CTAS_PER_SM) * num_sms()) / p.B);
  const long long nvec = (static_cast<long long>(p.V) + VE - 1) / VE;
  const long long cd_walk = chain ? (nvec + DRAW_MAX_VECTORS - 1) / DRAW_MAX_VECTORS
                                  : (static_cast<long long>(p.V) + NT * NT - 1) / (NT * NT);
  int CD = static_cast<int>(std::min<long long>(MAX_CLUSTER, std::max(cd_walk, std::min(cd_size, cd_wave))));
  for (;;) {
    const int per_d = (p.V + CD - 1) / CD;
    const int slice_d = (per_d + VE - 1) / VE * VE;
    if (chain ? (slice_d + VE - 1) / VE > DRAW_MAX_VECTORS : slice_d > NT * NT)
      return fail(SPEC_ERR_ARG, "vocabulary too large");
    const auto range = [&](int sl) { return ((sl + VE - 1) / VE + NWARP - 1) / NWARP * VE; };
    // the walk buffer: a warp range (tree draw), or the vector masses of a
    // CTA slice and the partials' masses of a row (chain draw)
    const int wlen = std::max({range(slice_d), range(g->slice), (slice_d + VE - 1) / VE, g->C * NCW});
    g->slice_d = slice_d;
    g->wbuf_off = base;
    g->smem_b = base + 4 * wlen;
    int nclus = 0;
    if ((st = occupancy(g->fb, g->smem_b, CD, &nclus))) return st;
    if (nclus > 0) break;
    if (CD == 1) return fail(SPEC_ERR_UNSUPPORTED, "no cluster fits on the device");
    CD = CD > 8 ? 8 : CD / 2;
  }
  g->CD = CD;
  return SPEC_OK;
}

// The two launches of a call: A (row statistics, persistent grid) then B
// (per-sequence decisions and outputs) as a programmatic dependent of A.
// One-shot measurement hook (spec_arm_rows_event): recorded on the stream
// between the two launches of the next call on this host thread.
thread_local cudaEvent_t g_rows_event = nullptr;
// One-shot measurement hook (spec_arm_timer): device stamps of the next call.
thread_local unsigned long long *g_timer = nullptr;

int launch(Params &p, const Geometry &g, cudaStream_t stream, float4 *partials, int32_t *status) {
  const cudaEvent_t ev_rows = g_rows_event;
  g_rows_event = nullptr;
  p.timer = g_timer;
  g_timer = nullptr;
  p.tickets = tickets_of(status);
  p.nshard = g.nshard;
  p.C = g.C;
  p.slice = g.slice;
  p.slice_d = g.slice_d;
  p.wbuf_off = g.wbuf_off;
  p.tile = g.tile;
  p.stages = g.stages;
  p.partials = partials;
  p.status = status;
  const bool argmax = p.kind == KIND_GREEDY_CHAIN || p.kind == KIND_TREE;
  cudaError_t e;
  {
    // a programmatic dependent of whatever precedes it on the stream: its
    // CTAs may be set up early, and it waits for that work before reading
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g.grid_a), 1, 1);
    cfg.blockDim = dim3(NT_ROW, 1, 1);
    cfg.dynamicSmemBytes = g.smem_a;
    cfg.stream = stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    e = launch_kernel(&cfg, g.fa, args);
    if (e != cudaSuccess) return cuda_fail(e, "row kernel launch");
  }
  if (ev_rows && (e = cudaEventRecord(ev_rows, stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = g.smem_b;
  cfg.stream = stream;
  if (argmax) {
    int per_sm = 0, st;
    if ((st = occupancy(g.fb, g.smem_b, 0, &per_sm))) return st;
    cfg.gridDim = dim3(static_cast<unsigned>(p.B), 1, 1);
  } else {
    cfg.gridDim = dim3(static_cast<unsigned>(p.B * g.CD), 1, 1);
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = g.CD;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void *args[] = {&p};
  e = launch_kernel(&cfg, g.fb, args);
  if (e != cudaSuccess) {
    // the decision kernel puts the tickets back to zero; without it, do it here
    cudaMemsetAsync(p.tickets, 0, sizeof(int) * NSHARD * TICKET_STRIDE, stream);
    return cuda_fail(e, "decision kernel launch");
  }
  return SPEC_OK;
}

// The step on this stream's workspace.
int run_step(Params &p, int dtype, bool tma, cudaStream_t stream, Workspace **ws_out) {
  Geometry g;
  int st = plan(p, dtype, tma, &g);
  if (st) return st;
  Workspace *w = nullptr;
  if ((st = get_ws(stream, static_cast<size_t>(g.nitems) * NCW, &w))) return st;
  *ws_out = w;
  return launch(p, g, stream, w->partials, w->status);
}

// The step on scratch the caller provides (partials with room for cap_parts
// entries, and a status word); nothing is allocated.  Used by the
// no-allocation entry point below.
int run_step_on(Params &p, int dtype, bool tma, cudaStream_t stream, float4 *partials,
                size_t cap_parts, int32_t *status) {
  Geometry g;
  int st = plan(p, dtype, tma, &g);
  if (st) return st;
  if (static_cast<size_t>(g.nitems) * NCW > cap_parts)
    return fail(SPEC_ERR_ARG, "call too large for the fixed scratch of spec_verify_noalloc: "
                              "B * (K+1) * ceil(V * element size / 16384) must not exceed " +
                                  std::to_string(cap_parts / NCW));
  return launch(p, g, stream, partials, status);
}

int check_common(const void *zt, int B, int V, int dtype) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_DTYPE, "dtype must be SPEC_F32 or SPEC_BF16");
  if (B < 0) return fail(SPEC_ERR_ARG, "B must be >= 0");
  if (V < 1) return fail(SPEC_ERR_ARG, "V must be >= 1");
  if (B > 0 && !zt) return fail(SPEC_ERR_ARG, "target_logits is NULL");
  return SPEC_OK;
}

// Chain verification.  point: q is the point mass at each draft token (no
// draft rows); counts: drafts per sequence [B] (NULL: K).
int verify_chain(const void *zt, const void *zd, const int32_t *x, int B, int K, int V, int dtype,
                 float T, uint64_t seed, int32_t *out_tokens, int32_t *out_n, float *row_max,
                 float *row_sumexp, spec_stats_t *stats, void *stream_ptr, const int32_t *counts = nullptr,
                 bool point = false) {
  int st = check_common(zt, B, V, dtype);
  if (st) return st;
  if (K < 0 || K > SPEC_MAX_DRAFTS) return fail(SPEC_ERR_ARG, "K out of range [0, 255]");
  if (!(T >= 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_ARG, "temperature must be finite and >= 0");
  const double cd = T > 0.f ? 1.4426950408889634 / static_cast<double>(T) : 0.0;
  if (T > 0.f && !(cd < 1e30)) return fail(SPEC_ERR_ARG, "temperature too small");
  if (B == 0) return SPEC_OK;
  if (!out_tokens || !out_n) return fail(SPEC_ERR_ARG, "output pointer is NULL");
  if (K > 0 && !x) return fail(SPEC_ERR_ARG, "draft_tokens is NULL");
  if (K > 0 && T > 0.f && !zd && !point) return fail(SPEC_ERR_ARG, "draft_logits is NULL with T > 0");
  if (static_cast<long long>(B) * (K + 1) * MAX_CLUSTER > INT_MAX) return fail(SPEC_ERR_ARG, "B*(K+1) too large");

  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool sample = T > 0.f;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(zt) &&
                   (!sample || K == 0 || point || aligned16(zd));
  Params p = {};
  p.zt = zt;
  p.zd = point ? nullptr : zd;
  p.tokens = x;
  p.parent = nullptr;
  p.counts = counts;
  p.point = point && sample;
  p.B = B;
  p.K = K;
  p.V = V;
  p.J = K + 1;
  p.kind = sample ? KIND_SAMPLE : KIND_GREEDY_CHAIN;
  p.c = static_cast<float>(cd);
  p.seed = seed;
  p.njobs = B * (K + 1);
  p.max_depth = 0;
  p.out_tokens = out_tokens;
  p.out_n = out_n;
  p.out_row_max = row_max;
  p.out_row_sumexp = row_sumexp;
  p.stats = reinterpret_cast<Stats *>(stats);
  Workspace *w = nullptr;
  return run_step(p, dtype, tma, static_cast<cudaStream_t>(stream_ptr), &w);
}

int tree_depth_host(const int32_t *parent, int N) {
  if (!parent || N < 1 || parent[0] != -1) return -1;
  std::vector<int> depth(N, 0);
  int D = 0;
  for (int c = 1; c < N; ++c) {
    if (parent[c] < 0 || parent[c] >= c) return -1;
    depth[c] = depth[parent[c]] + 1;
    D = std::max(D, depth[c]);
  }
  return D;
}


// ------------------------------------------------------------ EAGLE-2
int check_topk_args(int R, int V, int dtype, float T, int k) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_DTYPE, "dtype must be SPEC_F32 or SPEC_BF16");
  if (R < 0) return fail(SPEC_ERR_ARG, "row count must be >= 0");
  if (V < 1) return fail(SPEC_ERR_ARG, "V must be >= 1");
  if (k < 1 || k > SPEC_MAX_TOPK || k > V) return fail(SPEC_ERR_ARG, "need 1 <= k <= min(V, 32)");
  if (!(T > 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_ARG, "temperature must be finite and > 0");
  const double c = 1.4426950408889634 / static_cast<double>(T);
  if (!(c < 1e30)) return fail(SPEC_ERR_ARG, "temperature too small");
  return SPEC_OK;
}

// One launch of the top-k kernel (a programmatic dependent of earlier work):
// G CTAs per row in one cluster, each a contiguous slice of at least 32 KB,
// G a power of two up to 8 giving about one wave of 1.5 CTAs (of 512
// threads) per SM; rows enough for that wave take one CTA each.
int launch_topk(TopkParams &p, int dtype, cudaStream_t stream) {
  p.timer = g_timer;
  g_timer = nullptr;
  const size_t esz = dtype == SPEC_F32 ? 4 : 2;
  const bool vec = aligned16(p.z) && (static_cast<size_t>(p.V) * esz) % 16 == 0;
  const void *fn = dtype == SPEC_F32
                       ? (vec ? reinterpret_cast<const void *>(&topk_kernel<0, true>)
                              : reinterpret_cast<const void *>(&topk_kernel<0, false>))
                       : (vec ? reinterpret_cast<const void *>(&topk_kernel<1, true>)
                              : reinterpret_cast<const void *>(&topk_kernel<1, false>));
  const long long want = (3LL * num_sms() / 2 + p.R - 1) / p.R;
  const long long by_size = std::max<long long>(1, static_cast<long long>(p.V) * esz / 32768);
  int G = static_cast<int>(std::min<long long>({static_cast<long long>(TOPK_MAX_CLUSTER), want, by_size}));
  G = env_int("SPEC_TOPK_CLUSTER", G, 1, TOPK_MAX_CLUSTER);
  int pow2 = 1;
  while (pow2 * 2 <= G) pow2 *= 2;
  G = pow2;
  if (static_cast<long long>(p.R) * G > INT_MAX) return fail(SPEC_ERR_ARG, "too many rows");
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = G;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.R * G), 1, 1);
  cfg.blockDim = dim3(TOPK_NT, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void *args[] = {&p};
  cudaError_t e = launch_kernel(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "topk_kernel launch");
  return SPEC_OK;
}

int launch_eagle(const void *fn, EagleParams &p, int grid, int smem, cudaStream_t stream, const char *what) {
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  void *args[] = {&p};
  cudaError_t e = launch_kernel(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return SPEC_OK;
}
}  // namespace
}  // namespace spec

using namespace spec;

extern "C" {

int spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                int B, int K, int V, int dtype, float temperature, uint64_t seed,
                int32_t *out_tokens, int32_t *out_n_accepted, void *stream) {
  NvtxRange nvtx_range("spec_verify");
  return verify_chain(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed,
                      out_tokens, out_n_accepted, nullptr, nullptr, nullptr, stream);
}

int spec_verify_points(const void *target_logits, const int32_t *draft_tokens, const int32_t *draft_counts, int B,
                       int K, int V, int dtype, float temperature, uint64_t seed, int32_t *out_tokens,
                       int32_t *out_n_accepted, void *stream) {
  NvtxRange nvtx_range("spec_verify_points");
  return verify_chain(target_logits, nullptr, draft_tokens, B, K, V, dtype, temperature, seed, out_tokens,
                      out_n_accepted, nullptr, nullptr, nullptr, stream, draft_counts, true);
}

int spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                   int B, int K, int V, int dtype, float temperature, uint64_t seed,
                   int32_t *out_tokens, int32_t *out_n_accepted, float *out_row_max,
                   float *out_row_sumexp, spec_stats_t *stats, void *stream) {
  NvtxRange nvtx_range("spec_verify_ex");
  return verify_chain(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed,
                      out_tokens, out_n_accepted, out_row_max, out_row_sumexp, stats, stream);
}

// Greedy tree verification; parent_stride 0: one tree [N] for the batch,
// N: tree b at parent + b * N.
static int tree_greedy_impl(const void *target_logits, const int32_t *parent, int parent_stride,
                            const int32_t *node_tokens, int B, int N, int V, int dtype,
                            int max_depth, int32_t *out_path, int32_t *out_len, void *stream_ptr) {
  int st = check_common(target_logits, B, V, dtype);
  if (st) return st;
  if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_ARG, "N out of range [1, 1024]");
  if (max_depth < 0 || max_depth >= N) return fail(SPEC_ERR_ARG, "max_depth out of range [0, N)");
  if (B == 0) return SPEC_OK;
  if (!parent || !node_tokens || !out_path || !out_len) return fail(SPEC_ERR_ARG, "NULL pointer");
  if (static_cast<long long>(B) * N * MAX_CLUSTER > INT_MAX) return fail(SPEC_ERR_ARG, "B*N too large");
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(target_logits);
  Params p = {};
  p.zt = target_logits;
  p.tokens = node_tokens;
  p.parent = parent;
  p.parent_stride = parent_stride;
  p.B = B;
  p.K = N;
  p.V = V;
  p.J = N;
  p.kind = KIND_TREE;
  p.njobs = B * N;
  p.max_depth = max_depth;
  p.out_tokens = out_path;
  p.out_n = out_len;
  Workspace *w = nullptr;
  return run_step(p, dtype, tma, static_cast<cudaStream_t>(stream_ptr), &w);
}

// Stochastic tree verification; parent_stride as for tree_greedy_impl.
static int tree_sample_impl(const void *target_logits, const void *draft_logits, const int32_t *parent,
                            int parent_stride, const int32_t *node_tokens, int B, int N, int V, int dtype,
                            float temperature, uint64_t seed, int max_depth, int32_t *out_path,
                            int32_t *out_len, void *stream_ptr) {
  const float T = temperature;
  if (!(T >= 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_ARG, "temperature must be finite and >= 0");
  if (T == 0.f)  // greedy matching of the same tree
    return tree_greedy_impl(target_logits, parent, parent_stride, node_tokens, B, N, V, dtype, max_depth,
                            out_path, out_len, stream_ptr);
  int st = check_common(target_logits, B, V, dtype);
  if (st) return st;
  const double cd = 1.4426950408889634 / static_cast<double>(T);
  if (!(cd < 1e30)) return fail(SPEC_ERR_ARG, "temperature too small");
  if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_ARG, "N out of range [1, 1024]");
  if (max_depth < 0 || max_depth >= N) return fail(SPEC_ERR_ARG, "max_depth out of range [0, N)");
  if (B == 0) return SPEC_OK;
  if (!parent || !node_tokens || !out_path || !out_len || !draft_logits)
    return fail(SPEC_ERR_ARG, "NULL pointer");
  if (static_cast<long long>(B) * N * MAX_CLUSTER > INT_MAX) return fail(SPEC_ERR_ARG, "B*N too large");
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(target_logits) &&
                   aligned16(draft_logits);
  Params p = {};
  p.zt = target_logits;
  p.zd = draft_logits;
  p.tokens = node_tokens;
  p.parent = parent;
  p.parent_stride = parent_stride;
  p.B = B;
  p.K = N;
  p.V = V;
  p.J = N;
  p.kind = KIND_TREE_SAMPLE;
  p.c = static_cast<float>(cd);
  p.seed = seed;
  p.njobs = B * N;
  p.max_depth = max_depth;
  p.out_tokens = out_path;
  p.out_n = out_len;
  Workspace *w = nullptr;
  return run_step(p, dtype, tma, static_cast<cudaStream_t>(stream_ptr), &w);
}

int spec_verify_tree_greedy(const void *target_logits, const int32_t *parent, const int32_t *node_tokens,
                            int B, int N, int V, int dtype, int max_depth, int32_t *out_path,
                            int32_t *out_len, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_tree_greedy");
  return tree_greedy_impl(target_logits, parent, 0, node_tokens, B, N, V, dtype, max_depth, out_path, out_len,
                          stream_ptr);
}

int spec_verify_trees_greedy(const void *target_logits, const int32_t *parents, const int32_t *node_tokens,
                             int B, int N, int V, int dtype, int max_depth, int32_t *out_path,
                             int32_t *out_len, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_trees_greedy");
  return tree_greedy_impl(target_logits, parents, N, node_tokens, B, N, V, dtype, max_depth, out_path, out_len,
                          stream_ptr);
}

int spec_verify_tree(const void *target_logits, const void *draft_logits, const int32_t *parent,
                     const int32_t *node_tokens, int B, int N, int V, int dtype, float temperature,
                     uint64_t seed, int max_depth, int32_t *out_path, int32_t *out_len, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_tree");
  return tree_sample_impl(target_logits, draft_logits, parent, 0, node_tokens, B, N, V, dtype, temperature, seed,
                          max_depth, out_path, out_len, stream_ptr);
}

int spec_verify_trees(const void *target_logits, const void *draft_logits, const int32_t *parents,
                      const int32_t *node_tokens, int B, int N, int V, int dtype, float temperature,
                      uint64_t seed, int max_depth, int32_t *out_path, int32_t *out_len, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_trees");
  return tree_sample_impl(target_logits, draft_logits, parents, N, node_tokens, B, N, V, dtype, temperature, seed,
                          max_depth, out_path, out_len, stream_ptr);
}

int spec_tree_max_depth(const int32_t *parent_host, int N) {
  const int D = tree_depth_host(parent_host, N);
  if (D < 0) return fail(-SPEC_ERR_PARENT, "parent[] is not a tree");
  return D;
}

int spec_tree_mask(const int32_t *parent, int B, int N, uint32_t *out_mask, int32_t *out_depth,
                   void *stream_ptr) {
  NvtxRange nvtx_range("spec_tree_mask");
  if (B < 0) return fail(SPEC_ERR_ARG, "B must be >= 0");
  if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_ARG, "N out of range [1, 1024]");
  if (B == 0) return SPEC_OK;
  if (!parent || !out_mask || !out_depth) return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  int st = get_ws(stream, 1, &w);
  if (st) return st;
  const int W = (N + 31) / 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.stream = stream;
  int32_t *status = w->status;
  void *args[] = {(void *)&parent, (void *)&N, (void *)&W, (void *)&out_mask, (void *)&out_depth, (void *)&status};
  cudaError_t e = launch_kernel(&cfg, reinterpret_cast<const void *>(&tree_mask_kernel), args);
  if (e != cudaSuccess) return cuda_fail(e, "tree_mask_kernel launch");
  return SPEC_OK;
}

int spec_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B, int L, int n_min, int n_max,
                       int min_hits, int K, int32_t *out_draft, int32_t *out_count, void *stream_ptr) {
  NvtxRange nvtx_range("spec_ngram_propose");
  if (B < 0 || L < 0) return fail(SPEC_ERR_ARG, "B and L must be >= 0");
  if (n_min < 1 || n_max < n_min || n_max > SPEC_MAX_NGRAM)
    return fail(SPEC_ERR_ARG, "need 1 <= n_min <= n_max <= 64");
  if (min_hits < 1) return fail(SPEC_ERR_ARG, "min_hits must be >= 1");
  if (K < 0 || K > SPEC_MAX_DRAFTS) return fail(SPEC_ERR_ARG, "K out of range [0, 255]");
  if (B == 0) return SPEC_OK;
  if (!lengths || !out_count || (K > 0 && !out_draft) || (L > 0 && !tokens))
    return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int mode = min_hits == 1 ? NGRAM_MAXKEY
                   : n_max - n_min < NGRAM_REG_BINS ? NGRAM_REGHIST : NGRAM_SMEMHIST;
  const bool vec = L % 4 == 0 && aligned16(tokens);
  // CTAs per sequence: one round of loads each (4096 positions) if the
  // batch then fits in about one wave of resident CTAs (up to 1.25 waves),
  // else as many as one wave holds: the call is a chain of dependent memory
  // round trips, and a second round or a second wave each add one
  int per_sm = 0;
  {
    const void *probe = vec ? reinterpret_cast<const void *>(&ngram_kernel<true, NGRAM_MAXKEY, true>)
                            : reinterpret_cast<const void *>(&ngram_kernel<false, NGRAM_MAXKEY, true>);
    if (mode == NGRAM_REGHIST)
      probe = vec ? reinterpret_cast<const void *>(&ngram_kernel<true, NGRAM_REGHIST, true>)
                  : reinterpret_cast<const void *>(&ngram_kernel<false, NGRAM_REGHIST, true>);
    else if (mode == NGRAM_SMEMHIST)
      probe = vec ? reinterpret_cast<const void *>(&ngram_kernel<true, NGRAM_SMEMHIST, true>)
                  : reinterpret_cast<const void *>(&ngram_kernel<false, NGRAM_SMEMHIST, true>);
    int st0 = occupancy(probe, 0, 0, &per_sm);
    if (st0) return st0;
  }
  const long long slots = std::max(1LL, static_cast<long long>(per_sm) * num_sms());
  const long long g_round = std::max(1, (L + 4095) / 4096);
  long long G = static_cast<long long>(B) * g_round * 4 <= slots * 5 ? g_round
                                                                      : std::max(1LL, std::min(g_round, slots / B));
  G = env_int("SPEC_NGRAM_CTAS", static_cast<int>(G), 1, 1 << 16);
  if (static_cast<long long>(B) * G > INT_MAX) return fail(SPEC_ERR_ARG, "B too large");
  const size_t part_bytes = static_cast<size_t>(B) * G *
                            (mode == NGRAM_MAXKEY ? 8 : 8 * static_cast<size_t>(n_max - n_min + 1));
  Workspace *w = nullptr;
  int st = get_ws(stream, (part_bytes + 15) / 16, &w);
  if (st) return st;
  if (w->ngram_cap < static_cast<size_t>(B)) {
    std::lock_guard<std::mutex> lock(g_mu);
    cudaError_t e;
    if (w->ngram_done) {
      e = cudaFree(w->ngram_done);  // synchronises the device: no call still uses it
      w->ngram_done = nullptr;
      w->ngram_cap = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree(ngram counters)");
    }
    if ((e = cudaMalloc(&w->ngram_done, sizeof(int) * B)) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc(ngram counters)");
    if ((e = cudaMemsetAsync(w->ngram_done, 0, sizeof(int) * B, stream)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync(ngram counters)");
    w->ngram_cap = B;
  }
  // G <= 8: the sequence's CTAs form a cluster and combine on chip
  const bool cl = G <= NGRAM_MAX_CLUSTER;
#define SPEC_NGRAM_FNS(V, C)                                                 \
  {reinterpret_cast<const void *>(&ngram_kernel<V, NGRAM_MAXKEY, C>),        \
   reinterpret_cast<const void *>(&ngram_kernel<V, NGRAM_REGHIST, C>),       \
   reinterpret_cast<const void *>(&ngram_kernel<V, NGRAM_SMEMHIST, C>)}
  static const void *const fns[2][2][3] = {{SPEC_NGRAM_FNS(false, false), SPEC_NGRAM_FNS(false, true)},
                                           {SPEC_NGRAM_FNS(true, false), SPEC_NGRAM_FNS(true, true)}};
#undef SPEC_NGRAM_FNS
  NgramParams p{tokens, lengths, B, L, n_min, n_max, min_hits, K, static_cast<int>(G), out_draft, out_count,
                w->status, w->partials, w->ngram_done};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl ? static_cast<unsigned>(G) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B * G), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void *args[] = {&p};
  cudaError_t e = launch_kernel(&cfg, fns[vec][cl][mode], args);
  if (e != cudaSuccess) return cuda_fail(e, "ngram_kernel launch");
  return SPEC_OK;
}

int spec_topk(const void *logits, int R, int V, int dtype, float temperature, int k, int32_t *out_tokens,
              float *out_prob, void *stream_ptr) {
  NvtxRange nvtx_range("spec_topk");
  int st = check_topk_args(R, V, dtype, temperature, k);
  if (st) return st;
  if (R == 0) return SPEC_OK;
  if (!logits || !out_tokens || !out_prob) return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  if ((st = get_ws(stream, 1, &w))) return st;
  TopkParams p{};
  p.z = logits;
  p.R = R;
  p.V = V;
  p.k = k;
  p.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  p.out_tok = out_tokens;
  p.out_prob = out_prob;
  p.F = 0;
  p.status = w->status;
  return launch_topk(p, dtype, stream);
}

int spec_eagle2_expand(const void *draft_logits, const int32_t *frontier, int B, int F, int V, int dtype,
                       float temperature, int k, int32_t *node_tokens, float *node_values, int32_t *node_parents,
                       int cap, int offset, int k_next, int32_t *out_frontier, void *stream_ptr) {
  NvtxRange nvtx_range("spec_eagle2_expand");
  if (B < 0 || F < 1) return fail(SPEC_ERR_ARG, "need B >= 0 and F >= 1");
  int st = check_topk_args(B, V, dtype, temperature, k);
  if (st) return st;
  if (static_cast<long long>(F) * k > SPEC_EAGLE_MAX_CANDIDATES)
    return fail(SPEC_ERR_ARG, "F * k above 4096");
  if (offset < 1 || static_cast<long long>(offset) + static_cast<long long>(F) * k > cap)
    return fail(SPEC_ERR_ARG, "need 1 <= offset and offset + F * k <= cap");
  if (k_next < 0 || k_next > F * k) return fail(SPEC_ERR_ARG, "need 0 <= k_next <= F * k");
  if (static_cast<long long>(B) * F > INT_MAX || static_cast<long long>(B) * cap > (1LL << 40))
    return fail(SPEC_ERR_ARG, "B * F too large");
  if (B == 0) return SPEC_OK;
  if (!draft_logits || !frontier || !node_tokens || !node_values || !node_parents ||
      (k_next > 0 && !out_frontier))
    return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  if ((st = get_ws(stream, 1, &w))) return st;
  TopkParams tp{};
  tp.z = draft_logits;
  tp.R = B * F;
  tp.V = V;
  tp.k = k;
  tp.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  tp.out_tok = node_tokens;
  tp.out_prob = node_values;
  tp.F = F;
  tp.cap = cap;
  tp.offset = offset;
  tp.frontier = frontier;
  tp.node_par = node_parents;
  tp.status = w->status;
  if ((st = launch_topk(tp, dtype, stream))) return st;
  EagleParams ep{};
  ep.B = B;
  ep.F = F;
  ep.k = k;
  ep.cap = cap;
  ep.offset = offset;
  ep.k_next = k_next;
  ep.frontier = frontier;
  ep.node_tok = node_tokens;
  ep.node_val = node_values;
  ep.node_par = node_parents;
  ep.out_next = out_frontier;
  ep.status = w->status;
  return launch_eagle(reinterpret_cast<const void *>(&expand_select_kernel), ep, B, 0, stream,
                      "expand_select_kernel launch");
}

int spec_eagle2_rerank(const float *node_values, const int32_t *node_parents, const int32_t *node_tokens, int B,
                       int M, int m, int32_t *out_parent, int32_t *out_tokens, int32_t *out_index,
                       void *stream_ptr) {
  NvtxRange nvtx_range("spec_eagle2_rerank");
  if (B < 0) return fail(SPEC_ERR_ARG, "B must be >= 0");
  if (M < 1 || M > SPEC_EAGLE_MAX_NODES) return fail(SPEC_ERR_ARG, "M out of range [1, 8192]");
  if (m < 0 || m > M - 1) return fail(SPEC_ERR_ARG, "need 0 <= m <= M - 1");
  if (B == 0) return SPEC_OK;
  if (!node_values || !node_parents || !node_tokens || !out_parent || !out_tokens || !out_index)
    return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  int st = get_ws(stream, 1, &w);
  if (st) return st;
  const void *fn = reinterpret_cast<const void *>(&rerank_kernel);
  const int smem = 20 * M + 4 * m;
  int per_sm = 0;
  if ((st = occupancy(fn, smem, 0, &per_sm))) return st;
  if (per_sm < 1) return fail(SPEC_ERR_UNSUPPORTED, "rerank kernel does not fit on an SM");
  EagleParams ep{};
  ep.B = B;
  ep.M = M;
  ep.m = m;
  ep.node_tok = const_cast<int32_t *>(node_tokens);
  ep.node_val = const_cast<float *>(node_values);
  ep.node_par = const_cast<int32_t *>(node_parents);
  ep.out_par = out_parent;
  ep.out_tok = out_tokens;
  ep.out_idx = out_index;
  ep.status = w->status;
  return launch_eagle(fn, ep, B, smem, stream, "rerank_kernel launch");
}

int spec_selftest_wait(void *stream_ptr) {
  NvtxRange nvtx_range("spec_selftest_wait");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  int st = get_ws(stream, 1, &w);
  if (st) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = stream;
  int32_t *status = w->status;
  void *args[] = {&status};
  cudaError_t e = launch_kernel(&cfg, reinterpret_cast<const void *>(&wait_selftest_kernel), args);
  if (e != cudaSuccess) return cuda_fail(e, "wait_selftest_kernel launch");
  return SPEC_OK;
}

int spec_debug_fail_launch(int n) {
  if (n < 0) return fail(SPEC_ERR_ARG, "n must be >= 0");
  g_fail_launch.store(n);
  return SPEC_OK;
}

int spec_arm_timer(unsigned long long *stamps) {
  g_timer = stamps;
  return SPEC_OK;
}

int spec_arm_rows_event(void *event) {
  g_rows_event = static_cast<cudaEvent_t>(event);
  return SPEC_OK;
}

}  // extern "C"

namespace spec {
namespace {
// Reads the device status word at `word` (after the stream has drained),
// clears it, and maps its bits to a status code.
int read_status_word(int32_t *word) {
  int32_t bits = 0;
  cudaError_t e;
  if ((e = cudaMemcpy(&bits, word, sizeof bits, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy(status)");
  if (bits == 0) return SPEC_OK;
  if ((e = cudaMemset(word, 0, sizeof(int32_t))) != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  if (bits & ST_TIMEOUT) return fail(SPEC_ERR_TIMEOUT, "a bounded wait on the device ran out");
  if (bits & ST_PARENT) return fail(SPEC_ERR_PARENT, "parent[] is not a tree of the given depth");
  if (bits & ST_LENGTH) return fail(SPEC_ERR_ARG, "lengths[b] outside [0, L]");
  return fail(SPEC_ERR_TOKEN_RANGE, "a draft or node token is outside [0, V)");
}
}  // namespace
}  // namespace spec

extern "C" {

int spec_get_status(void *stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  Workspace *w;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    w = find_ws(dev, stream, false);
  }
  if (!w || !w->status) return SPEC_OK;
  return read_status_word(w->status);
}

int spec_verify_host(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                     int B, int K, int V, int dtype, float temperature, uint64_t seed,
                     int32_t *out_tokens, int32_t *out_n_accepted, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_host");
  int st = check_common(target_logits, B, V, dtype);
  if (st) return st;
  if (K < 0 || K > SPEC_MAX_DRAFTS) return fail(SPEC_ERR_ARG, "K out of range [0, 255]");
  if (B == 0) return SPEC_OK;
  if (!out_tokens || !out_n_accepted) return fail(SPEC_ERR_ARG, "output pointer is NULL");
  const bool sample = temperature > 0.f;
  if (K > 0 && !draft_tokens) return fail(SPEC_ERR_ARG, "draft_tokens is NULL");
  if (K > 0 && sample && !draft_logits) return fail(SPEC_ERR_ARG, "draft_logits is NULL with T > 0");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const size_t esz = dtype == SPEC_F32 ? 4 : 2;
  auto up = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t bt = static_cast<size_t>(B) * (K + 1) * V * esz;
  const size_t bd = (sample && K > 0) ? static_cast<size_t>(B) * K * V * esz : 0;
  const size_t bx = static_cast<size_t>(B) * K * sizeof(int32_t);
  const size_t bo = static_cast<size_t>(B) * (K + 1) * sizeof(int32_t);
  const size_t bn = static_cast<size_t>(B) * sizeof(int32_t);
  const size_t total = up(bt) + up(bd) + up(bx) + up(bo) + up(bn);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  Workspace *w;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    w = find_ws(dev, stream, true);
    if (w->stage_cap < total) {
      if (w->stage) cudaFree(w->stage);
      w->stage = nullptr;
      w->stage_cap = 0;
      if ((e = cudaMalloc(&w->stage, total)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(staging)");
      w->stage_cap = total;
    }
  }
  unsigned char *d = w->stage;
  void *dzt = d;
  void *dzd = bd ? d + up(bt) : nullptr;
  int32_t *dx = bx ? reinterpret_cast<int32_t *>(d + up(bt) + up(bd)) : nullptr;
  int32_t *dout = reinterpret_cast<int32_t *>(d + up(bt) + up(bd) + up(bx));
  int32_t *dn = reinterpret_cast<int32_t *>(d + up(bt) + up(bd) + up(bx) + up(bo));
  if ((e = cudaMemcpyAsync(dzt, target_logits, bt, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync(target)");
  if (bd && (e = cudaMemcpyAsync(dzd, draft_logits, bd, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync(draft)");
  if (bx && (e = cudaMemcpyAsync(dx, draft_tokens, bx, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync(tokens)");
  if ((st = spec_verify(dzt, dzd, dx, B, K, V, dtype, temperature, seed, dout, dn, stream))) return st;
  if ((e = cudaMemcpyAsync(out_tokens, dout, bo, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync(out_tokens)");
  if ((e = cudaMemcpyAsync(out_n_accepted, dn, bn, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync(out_n)");
  return spec_get_status(stream_ptr);
}

const char *spec_error_string(int status) {
  switch (status < 0 ? -status : status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_ARG: return "SPEC_ERR_ARG";
    case SPEC_ERR_DTYPE: return "SPEC_ERR_DTYPE";
    case SPEC_ERR_ALIGN: return "SPEC_ERR_ALIGN";
    case SPEC_ERR_TOKEN_RANGE: return "SPEC_ERR_TOKEN_RANGE";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    case SPEC_ERR_PARENT: return "SPEC_ERR_PARENT";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    default: return "SPEC_ERR_UNKNOWN";
  }
}

const char *spec_last_error_message(void) { return g_last_error.c_str(); }

void spec_shutdown(void) {
  noalloc_forget();
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (Workspace *w : g_ws) {
    cudaSetDevice(w->device);
    if (w->status) cudaFree(w->status);
    if (w->partials) cudaFree(w->partials);
    if (w->stage) cudaFree(w->stage);
    if (w->ngram_done) cudaFree(w->ngram_done);
    delete w;
  }
  g_ws.clear();
  g_kc.clear();
  cudaSetDevice(cur);
}

}  // extern "C"

// ------------------------------------------------------------------------
// spec_verify_noalloc: spec_verify on a fixed scratch area compiled into the
// library.  Some callers cannot allocate device memory at call time: a
// serving engine that reserves nearly all HBM for its own pool at start-up,
// or a latency-critical loop that cannot pay for cudaMalloc/cudaFree (which
// may synchronise the whole device).  This entry point serves them: its
// scratch is the static array below, resident on every GPU that loads the
// library until the process exits, and the call allocates nothing.
namespace spec {
namespace {

// status word and item tickets (zero-initialised, and zero again after every
// call), then the row partials
constexpr size_t NOALLOC_MAX_PARTIALS = (size_t(1) << 16) * NCW;  // float4 entries: 8 MiB
constexpr size_t NOALLOC_PARTS_OFF = (CONTROL_BYTES + 255) / 256 * 256;
constexpr size_t NOALLOC_BYTES = NOALLOC_PARTS_OFF + NOALLOC_MAX_PARTIALS * sizeof(float4);
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
unsigned char *g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {nullptr};

void noalloc_forget() {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (auto &ptr : g_noalloc_ptr) ptr = nullptr;
}

// Device address of the scratch array on the current device, looked up once
// per device (the array's host-side name is only a stand-in).
int noalloc_scratch(unsigned char **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return fail(SPEC_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev] = static_cast<unsigned char *>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return SPEC_OK;
}

}  // namespace
}  // namespace spec

extern "C" int spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                   const int32_t *draft_tokens, int B, int K, int V, int dtype,
                                   float temperature, uint64_t seed, int32_t *out_tokens,
                                   int32_t *out_n_accepted, void *stream_ptr) {
  NvtxRange nvtx_range("spec_verify_noalloc");
  using namespace spec;
  int st = check_common(target_logits, B, V, dtype);
  if (st) return st;
  if (K < 0 || K > SPEC_MAX_DRAFTS) return fail(SPEC_ERR_ARG, "K out of range [0, 255]");
  const float T = temperature;
  if (!(T >= 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_ARG, "temperature must be finite and >= 0");
  const double cd = T > 0.f ? 1.4426950408889634 / static_cast<double>(T) : 0.0;
  if (T > 0.f && !(cd < 1e30)) return fail(SPEC_ERR_ARG, "temperature too small");
  if (B == 0) return SPEC_OK;
  if (!out_tokens || !out_n_accepted) return fail(SPEC_ERR_ARG, "output pointer is NULL");
  if (K > 0 && !draft_tokens) return fail(SPEC_ERR_ARG, "draft_tokens is NULL");
  if (K > 0 && T > 0.f && !draft_logits) return fail(SPEC_ERR_ARG, "draft_logits is NULL with T > 0");
  if (static_cast<long long>(B) * (K + 1) * MAX_CLUSTER > INT_MAX) return fail(SPEC_ERR_ARG, "B*(K+1) too large");
  unsigned char *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch))) return st;
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool sample = T > 0.f;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(target_logits) &&
                   (!sample || K == 0 || aligned16(draft_logits));
  Params p = {};
  p.zt = target_logits;
  p.zd = draft_logits;
  p.tokens = draft_tokens;
  p.B = B;
  p.K = K;
  p.V = V;
  p.J = K + 1;
  p.kind = sample ? KIND_SAMPLE : KIND_GREEDY_CHAIN;
  p.c = static_cast<float>(cd);
  p.seed = seed;
  p.njobs = B * (K + 1);
  p.out_tokens = out_tokens;
  p.out_n = out_n_accepted;
  return run_step_on(p, dtype, tma, static_cast<cudaStream_t>(stream_ptr),
                     reinterpret_cast<float4 *>(scratch + NOALLOC_PARTS_OFF), NOALLOC_MAX_PARTIALS,
                     reinterpret_cast<int32_t *>(scratch));
}

extern "C" int spec_noalloc_get_status(void *stream_ptr) {
  using namespace spec;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned char *scratch = nullptr;
  int st = noalloc_scratch(&scratch);
  if (st) return st;
  return read_status_word(reinterpret_cast<int32_t *>(scratch));
}

extern "C" int spec_debug_noalloc_status(int bits) {
  using namespace spec;
  unsigned char *scratch = nullptr;
  int st = noalloc_scratch(&scratch);
  if (st) return st;
  int32_t cur = 0;
  cudaError_t e;
  if ((e = cudaMemcpy(&cur, scratch, sizeof cur, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy(status)");
  cur |= bits & (ST_TOKEN | ST_PARENT | ST_TIMEOUT);
  if ((e = cudaMemcpy(scratch, &cur, sizeof cur, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy(status)");
  return SPEC_OK;
}
