// Host side of libspec_verify.so: argument validation, launch geometry
// (cluster size, slices, tiles, stages), per-stream workspaces and the C ABI
// declared in include/spec_verify.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.cuh"
#include "spec_verify.h"

namespace spec {
namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string &msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return SPEC_ERR_CUDA;
}

// ------------------------------------------------------------ workspaces
// Per (device, stream): [status][ticket B][first_rej B][seq_err B][cand B*J]
// plus a staging area for the host-buffer entry point.
struct Workspace {
  int device = -1;
  cudaStream_t stream = nullptr;
  int32_t *status = nullptr;  // 1 word, never reallocated
  int32_t *ints = nullptr;
  size_t cap_seq = 0, cap_cand = 0;
  unsigned char *stage = nullptr;
  size_t stage_cap = 0;
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

// Returns SPEC_OK and the workspace holding at least B sequences and B*J jobs.
int get_ws(cudaStream_t stream, size_t B, size_t J, Workspace **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace *w = find_ws(dev, stream, true);
  if (!w->status) {
    e = cudaMalloc(&w->status, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
    e = cudaMemsetAsync(w->status, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  }
  const size_t need_seq = std::max<size_t>(B, 1), need_cand = std::max<size_t>(B * J, 1);
  if (w->cap_seq < need_seq || w->cap_cand < need_cand) {
    const size_t seq = std::max(need_seq, w->cap_seq), cand = std::max(need_cand, w->cap_cand);
    if (w->ints) {
      e = cudaFree(w->ints);  // synchronises the device: no call still uses it
      w->ints = nullptr;
      w->cap_seq = w->cap_cand = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    int32_t *p = nullptr;
    e = cudaMalloc(&p, sizeof(int32_t) * (3 * seq + cand));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    // ticket = 0, first_rej = "none" (0x7F7F7F7F), seq_err = 0, cand = 0
    if ((e = cudaMemsetAsync(p, 0, sizeof(int32_t) * seq, stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(p + seq, 0x7F, sizeof(int32_t) * seq, stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(p + 2 * seq, 0, sizeof(int32_t) * (seq + cand), stream)) != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(e, "cudaMemsetAsync(workspace)");
    }
    w->ints = p;
    w->cap_seq = seq;
    w->cap_cand = cand;
  }
  *out = w;
  return SPEC_OK;
}

void bind_ws(Params &p, const Workspace *w) {
  p.status = w->status;
  p.ticket = w->ints;
  p.first_rej = w->ints + w->cap_seq;
  p.seq_err = w->ints + 2 * w->cap_seq;
  p.cand = w->ints + 3 * w->cap_seq;
}

// ------------------------------------------------------------ geometry
constexpr int SLICE_TARGET_BYTES = 16 * 1024;  // vocabulary bytes per row and CTA
constexpr int DEFAULT_STAGES = 4;               // tile ring depth

int env_int(const char *name, int dflt, int lo, int hi) {
  const char *v = std::getenv(name);
  if (!v || !*v) return dflt;
  const int x = std::atoi(v);
  return (x >= lo && x <= hi) ? x : dflt;
}

struct KernelCache {
  const void *fn;
  int device;
  int smem_set;
  int C, smem, max_clusters;  // last occupancy query
};
std::vector<KernelCache> g_kc;

cudaLaunchConfig_t cluster_config(const void *fn, int C, int grid_clusters, int smem,
                                  cudaStream_t stream, cudaLaunchAttribute *attr) {
  (void)fn;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C * grid_clusters), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = C;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Sets the kernel's attributes once per device and returns how many clusters
// of size C with `smem` bytes can be resident at once (0: none).
int prepare_kernel(const void *fn, int C, int smem, int *max_clusters) {
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
    k.C = -1;
    g_kc.push_back(k);
    kc = &g_kc.back();
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
  }
  if (smem > kc->smem_set) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    kc->smem_set = smem;
    kc->C = -1;
  }
  if (kc->C != C || kc->smem != smem) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = cluster_config(fn, C, 1, smem, nullptr, &attr);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (e != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    kc->C = C;
    kc->smem = smem;
    kc->max_clusters = n;
  }
  *max_clusters = kc->max_clusters;
  return SPEC_OK;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

const void *pick_sample_kernel(int dtype, bool tma) {
  if (dtype == SPEC_F32)
    return tma ? reinterpret_cast<const void *>(&sample_kernel<0, true>)
               : reinterpret_cast<const void *>(&sample_kernel<0, false>);
  return tma ? reinterpret_cast<const void *>(&sample_kernel<1, true>)
             : reinterpret_cast<const void *>(&sample_kernel<1, false>);
}

const void *pick_argmax_kernel(int dtype, bool tma) {
  if (dtype == SPEC_F32)
    return tma ? reinterpret_cast<const void *>(&argmax_kernel<0, true>)
               : reinterpret_cast<const void *>(&argmax_kernel<0, false>);
  return tma ? reinterpret_cast<const void *>(&argmax_kernel<1, true>)
             : reinterpret_cast<const void *>(&argmax_kernel<1, false>);
}

// Launch geometry: cluster size C (CTAs sharing one row), slice per CTA,
// tile, ring depth, dynamic shared memory, clusters launched.
struct Geometry {
  int C, slice, tile, stages, smem, emit_off, ncl;
};

// Slices of about 16 KB per row and CTA (cluster size up to 16), tiles of
// NT threads x 2 vectors of 16 bytes, a ring of `stages` tiles (each stage
// holds `srows` rows), then as many clusters as can be resident, capped by
// the number of jobs.
int plan(const void *fn, int V, int dtype, int srows, int emit_bytes, long long njobs,
         Geometry *g) {
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const int VE = 16 / esz;
  const long long row_bytes = static_cast<long long>(V) * esz;
  int C = static_cast<int>(std::min<long long>(
      16, std::max<long long>(1, (row_bytes + SLICE_TARGET_BYTES - 1) / SLICE_TARGET_BYTES)));
  C = env_int("SPEC_VERIFY_CLUSTER", C, 1, 16);
  g->stages = env_int("SPEC_VERIFY_STAGES", DEFAULT_STAGES, 1, MAX_STAGES);
  g->tile = NT * VE * VECS_PER_THREAD;
  for (;;) {
    const int per = (V + C - 1) / C;
    g->slice = (per + VE - 1) / VE * VE;
    // the draw's per-thread chunk must fit one block-wide pass (slice <= NT^2)
    if (g->slice > NT * NT || (g->slice + g->tile - 1) / g->tile > MAX_TILES * 64)
      return fail(SPEC_ERR_ARG, "vocabulary too large (V <= 1048576)");
    g->emit_off = g->stages * srows * g->tile * esz;
    g->smem = g->emit_off + emit_bytes;
    int maxc = 0;
    int st = prepare_kernel(fn, C, g->smem, &maxc);
    if (st) return st;
    if (maxc > 0) {
      g->C = C;
      g->ncl = static_cast<int>(std::min<long long>(njobs, maxc));
      return SPEC_OK;
    }
    if (C == 1) return fail(SPEC_ERR_UNSUPPORTED, "no cluster of this size fits on the device");
    C = C > 8 ? 8 : C / 2;
  }
}

int launch(const void *fn, const Geometry &g, cudaStream_t stream, Params &p) {
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = cluster_config(fn, g.C, g.ncl, g.smem, stream, &attr);
  p.slice = g.slice;
  p.tile = g.tile;
  p.stages = g.stages;
  p.ncl = g.ncl;
  p.emit_off = g.emit_off;
  void *args[] = {&p};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return SPEC_OK;
}

int check_common(const void *zt, int B, int V, int dtype) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_DTYPE, "dtype must be SPEC_F32 or SPEC_BF16");
  if (B < 0) return fail(SPEC_ERR_ARG, "B must be >= 0");
  if (V < 1) return fail(SPEC_ERR_ARG, "V must be >= 1");
  if (B > 0 && !zt) return fail(SPEC_ERR_ARG, "target_logits is NULL");
  return SPEC_OK;
}

int verify_chain(const void *zt, const void *zd, const int32_t *x, int B, int K, int V, int dtype,
                 float T, uint64_t seed, int32_t *out_tokens, int32_t *out_n, float *row_max,
                 float *row_sumexp, spec_stats_t *stats, void *stream_ptr) {
  int st = check_common(zt, B, V, dtype);
  if (st) return st;
  if (K < 0 || K > SPEC_MAX_DRAFTS) return fail(SPEC_ERR_ARG, "K out of range [0, 255]");
  if (!(T >= 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_ARG, "temperature must be finite and >= 0");
  const double cd = T > 0.f ? 1.4426950408889634 / static_cast<double>(T) : 0.0;
  if (T > 0.f && !(cd < 1e30)) return fail(SPEC_ERR_ARG, "temperature too small");
  if (B == 0) return SPEC_OK;
  if (!out_tokens || !out_n) return fail(SPEC_ERR_ARG, "output pointer is NULL");
  if (K > 0 && !x) return fail(SPEC_ERR_ARG, "draft_tokens is NULL");
  if (K > 0 && T > 0.f && !zd) return fail(SPEC_ERR_ARG, "draft_logits is NULL with T > 0");
  if (static_cast<long long>(B) * (K + 1) > INT_MAX / 16) return fail(SPEC_ERR_ARG, "B*(K+1) too large");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool sample = T > 0.f;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(zt) &&
                   (!sample || K == 0 || aligned16(zd));
  const void *fn = sample ? pick_sample_kernel(dtype, tma) : pick_argmax_kernel(dtype, tma);
  const long long njobs = static_cast<long long>(B) * (K + 1);
  Geometry g;
  if ((st = plan(fn, V, dtype, sample && K > 0 ? 2 : 1, sample ? 0 : 8 * (2 * K + 2), njobs, &g)))
    return st;
  Workspace *w = nullptr;
  if ((st = get_ws(stream, B, K + 1, &w))) return st;

  Params p = {};
  p.zt = zt;
  p.zd = zd;
  p.tokens = x;
  p.parent = nullptr;
  p.B = B;
  p.K = K;
  p.V = V;
  p.J = K + 1;
  p.kind = sample ? KIND_SAMPLE : KIND_GREEDY_CHAIN;
  p.c = static_cast<float>(cd);
  p.seed = seed;
  p.njobs = static_cast<int>(njobs);
  p.max_depth = 0;
  p.out_tokens = out_tokens;
  p.out_n = out_n;
  p.out_row_max = row_max;
  p.out_row_sumexp = row_sumexp;
  p.stats = reinterpret_cast<Stats *>(stats);
  bind_ws(p, w);
  return launch(fn, g, stream, p);
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

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" {

int spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                int B, int K, int V, int dtype, float temperature, uint64_t seed,
                int32_t *out_tokens, int32_t *out_n_accepted, void *stream) {
  return verify_chain(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed,
                      out_tokens, out_n_accepted, nullptr, nullptr, nullptr, stream);
}

int spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                   int B, int K, int V, int dtype, float temperature, uint64_t seed,
                   int32_t *out_tokens, int32_t *out_n_accepted, float *out_row_max,
                   float *out_row_sumexp, spec_stats_t *stats, void *stream) {
  return verify_chain(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed,
                      out_tokens, out_n_accepted, out_row_max, out_row_sumexp, stats, stream);
}

int spec_verify_tree_greedy(const void *target_logits, const int32_t *parent,
                            const int32_t *node_tokens, int B, int N, int V, int dtype,
                            int max_depth, int32_t *out_path, int32_t *out_len, void *stream_ptr) {
  int st = check_common(target_logits, B, V, dtype);
  if (st) return st;
  if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_ARG, "N out of range [1, 1024]");
  if (max_depth < 0 || max_depth >= N) return fail(SPEC_ERR_ARG, "max_depth out of range [0, N)");
  if (B == 0) return SPEC_OK;
  if (!parent || !node_tokens || !out_path || !out_len) return fail(SPEC_ERR_ARG, "NULL pointer");
  if (static_cast<long long>(B) * N > INT_MAX / 16) return fail(SPEC_ERR_ARG, "B*N too large");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int esz = dtype == SPEC_F32 ? 4 : 2;
  const bool tma = (static_cast<long long>(V) * esz) % 16 == 0 && aligned16(target_logits);
  const int emit_smem = 17 * N + 64;
  const void *fn = pick_argmax_kernel(dtype, tma);
  const long long njobs = static_cast<long long>(B) * N;
  Geometry g;
  if ((st = plan(fn, V, dtype, 1, emit_smem, njobs, &g))) return st;
  Workspace *w = nullptr;
  if ((st = get_ws(stream, B, N, &w))) return st;
  Params p = {};
  p.zt = target_logits;
  p.tokens = node_tokens;
  p.parent = parent;
  p.B = B;
  p.K = N;
  p.V = V;
  p.J = N;
  p.kind = KIND_TREE;
  p.njobs = static_cast<int>(njobs);
  p.max_depth = max_depth;
  p.out_tokens = out_path;
  p.out_n = out_len;
  bind_ws(p, w);
  return launch(fn, g, stream, p);
}

int spec_tree_max_depth(const int32_t *parent_host, int N) {
  const int D = tree_depth_host(parent_host, N);
  if (D < 0) return fail(-SPEC_ERR_PARENT, "parent[] is not a tree");
  return D;
}

int spec_tree_mask(const int32_t *parent, int B, int N, uint32_t *out_mask, int32_t *out_depth,
                   void *stream_ptr) {
  if (B < 0) return fail(SPEC_ERR_ARG, "B must be >= 0");
  if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_ARG, "N out of range [1, 1024]");
  if (B == 0) return SPEC_OK;
  if (!parent || !out_mask || !out_depth) return fail(SPEC_ERR_ARG, "NULL pointer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  Workspace *w = nullptr;
  int st = get_ws(stream, 1, 1, &w);
  if (st) return st;
  const int W = (N + 31) / 32;
  tree_mask_kernel<<<B, NT, 0, stream>>>(parent, N, W, out_mask, out_depth, w->status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "tree_mask_kernel launch");
  return SPEC_OK;
}

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
  int32_t bits = 0;
  if ((e = cudaMemcpy(&bits, w->status, sizeof bits, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy(status)");
  if (bits == 0) return SPEC_OK;
  if ((e = cudaMemset(w->status, 0, sizeof(int32_t))) != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  if (bits & ST_TIMEOUT) return fail(SPEC_ERR_TIMEOUT, "a bounded wait on the device ran out");
  if (bits & ST_PARENT) return fail(SPEC_ERR_PARENT, "parent[] is not a tree of the given depth");
  return fail(SPEC_ERR_TOKEN_RANGE, "a draft or node token is outside [0, V)");
}

int spec_verify_host(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                     int B, int K, int V, int dtype, float temperature, uint64_t seed,
                     int32_t *out_tokens, int32_t *out_n_accepted, void *stream_ptr) {
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
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (Workspace *w : g_ws) {
    cudaSetDevice(w->device);
    if (w->status) cudaFree(w->status);
    if (w->ints) cudaFree(w->ints);
    if (w->stage) cudaFree(w->stage);
    delete w;
  }
  g_ws.clear();
  g_kc.clear();
  cudaSetDevice(cur);
}

}  // extern "C"
