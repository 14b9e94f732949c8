/*
 * spec_verify.h — C ABI of the GB300 (sm_103a) verification step of
 * speculative decoding.
 *
 * One library, libspec_verify.so, with hand-written CUDA kernels behind plain
 * C entry points: pointers, sizes and a CUDA stream passed as void*.  No
 * C++ types, no exceptions and no torch types cross this boundary.
 *
 * Pages this interface restates:
 *   [Oscine]  blog.oscine.io, "投机解码：让大模型「猜」着跑的数学魔术"
 *   [Anhtu]   anhtu.dev, "Speculative Decoding: Cách LLM Sinh Văn Bản Nhanh
 *             Gấp 2–3 Lần"
 *   [Infra53] infra-guide, "5.3 Medusa, EAGLE và MTP"
 *   [Glukhov] glukhov.org, "Спекулятивное декодирование: ускорение
 *             инференса LLM на 20–50%"
 *
 * Common conventions
 *   - Logit tensors are contiguous, row-major, vocabulary innermost, either
 *     IEEE fp32 (SPEC_F32) or bfloat16 (SPEC_BF16).  Rows are read once.
 *   - Every tensor argument is a DEVICE pointer owned by the caller unless a
 *     function says otherwise; the library never frees or keeps them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = the legacy
 *     default stream) unless stated otherwise.  Argument errors are reported
 *     by the return value before anything is launched.  Errors found on the
 *     device (a token id outside [0, V), a malformed tree) are recorded per
 *     stream and returned by spec_get_status(); the affected sequence's
 *     count output is set to -1 and its token outputs to -1.
 *   - The fast path reads logits with TMA bulk copies and needs 16-byte
 *     aligned logits pointers and V * element_size divisible by 16; other
 *     layouts are accepted and take a slower path with plain loads.
 *   - Each row must hold at least one finite logit.  -inf entries (masked
 *     vocabulary) are allowed; NaN and +inf are not.
 *   - The first kernel of a call is a programmatic dependent launch of
 *     whatever precedes it on the stream: its blocks may be set up while
 *     that work drains, and they wait for it to complete before reading
 *     anything, so stream order is unchanged.
 *   - The library keeps one grow-only device workspace per (device, stream)
 *     pair (a few ints per sequence).  Growing it calls cudaMalloc, so the
 *     first call of a new size on a stream should not be inside a CUDA graph
 *     capture.  Two calls that overlap on the GPU must use different streams.
 *     spec_shutdown() frees every workspace.
 *   - Identical inputs and seed give identical outputs, bit for bit.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = 1,          /* null pointer, size out of range, bad temperature */
  SPEC_ERR_DTYPE = 2,        /* unknown dtype code */
  SPEC_ERR_ALIGN = 3,        /* reserved: misaligned inputs take the slow path */
  SPEC_ERR_TOKEN_RANGE = 4,  /* (device) a draft/node token outside [0, V) */
  SPEC_ERR_CUDA = 5,         /* a CUDA runtime error; see spec_last_error_message */
  SPEC_ERR_TIMEOUT = 6,      /* (device) a bounded wait ran out */
  SPEC_ERR_PARENT = 7,       /* parent[] is not a tree: parent[0] != -1 or parent[c] >= c */
  SPEC_ERR_UNSUPPORTED = 8   /* no usable GPU / cluster launch not possible */
};

/* Logit element types. */
enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

/* Size limits. */
#define SPEC_MAX_DRAFTS 255      /* K of a chain */
#define SPEC_MAX_TREE_NODES 1024 /* N of a tree */
#define SPEC_MAX_NGRAM 64        /* n_max of the n-gram drafter */
#define SPEC_MAX_TOPK 32         /* k of spec_topk / spec_eagle2_expand */
#define SPEC_EAGLE_MAX_CANDIDATES 4096 /* F * k of one expansion step */
#define SPEC_EAGLE_MAX_NODES 8192      /* M of spec_eagle2_rerank */

/* Counters a caller may ask spec_verify_ex to accumulate (device memory,
 * zeroed by the caller, added to atomically by every call that receives it).
 * They mirror the acceptance monitoring the pages recommend ([Glukhov]
 * §"Мониторинг в производстве": acceptance rate per request). */
typedef struct {
  unsigned long long sequences;          /* sequences verified without error */
  unsigned long long accepted;           /* sum of n_accepted */
  unsigned long long bonus;              /* sequences that accepted all K and drew a bonus */
  unsigned long long resampled;          /* sequences that stopped at a reject */
  unsigned long long residual_fallbacks; /* rejects whose residual mass was 0 in fp32 */
  unsigned long long errors;             /* sequences with an out-of-range token */
  unsigned long long near_boundary;      /* sequences with a decision near its boundary: an
                                            acceptance test with |u - p/q| <= 1e-5 max(p/q, 2^-24),
                                            or a draw whose t = u Z lies within 1e-5 Z of either end
                                            of the drawn token's CDF interval (fp32, as computed);
                                            such decisions are where another rounding of the same
                                            arithmetic could choose differently */
} spec_stats_t;

/*
 * spec_verify — chain verification of B sequences with K drafts each.
 *
 * For temperature T > 0 ([Oscine] §"验收标准的精确数学", eq. α(x);
 * §"拒绝之后怎么办？——残差分布", eq. p_resid; §"多 Token 验证：左到右，遇错即停"):
 *   p_i = softmax(target_logits[b, i, :] / T), i = 0..K,
 *   q_i = softmax(draft_logits[b, i, :] / T),  i = 0..K-1;
 *   draft x_i = draft_tokens[b, i] is accepted iff u_i < p_i(x_i) / q_i(x_i),
 *   scanning i = 0, 1, ... and stopping at the first reject j; the token at j
 *   is then drawn from norm(max(0, p_j - q_j)); if all K are accepted a bonus
 *   token is drawn from p_K ([Anhtu] §"Toán học của sự miễn phí").
 * For T == 0 the rule is greedy matching ([Infra53] §9.1): x_i is kept iff it
 * equals argmax p_i (lowest index on ties); the first mismatch emits
 * argmax p_j, a full match emits argmax p_K.  draft_logits is not read.
 *
 * Uniforms: u = (w >> 8) * 2^-24, w = word 0 of Philox4x32-10 with key
 * (seed mod 2^32, seed >> 32) and counter (b, position, slot, 0); slot 0 is
 * the acceptance test at position i, slot 1 the residual draw at position j
 * or the bonus draw at position K.  Draws invert the CDF in vocabulary order
 * (smallest v with C(v) > u * Z).
 *
 * Arguments
 *   target_logits   [B, K+1, V], dtype
 *   draft_logits    [B, K, V], dtype; may be NULL iff T == 0 or K == 0
 *   draft_tokens    [B, K] int32; may be NULL iff K == 0
 *   B >= 0 (B == 0 is a no-op), 0 <= K <= SPEC_MAX_DRAFTS, V >= 1
 *   dtype           SPEC_F32 or SPEC_BF16
 *   temperature     T >= 0, finite
 *   seed            64-bit Philox key
 *   out_tokens      [B, K+1] int32: accepted drafts, then the new token,
 *                   then -1 padding
 *   out_n_accepted  [B] int32: number of accepted drafts n (0..K), -1 on a
 *                   device-detected error in that sequence
 *   stream          cudaStream_t as void*
 * Returns SPEC_OK or an error code (nothing is launched on an error).
 */
int spec_verify(const void *target_logits, const void *draft_logits,
                const int32_t *draft_tokens, int B, int K, int V, int dtype,
                float temperature, uint64_t seed, int32_t *out_tokens,
                int32_t *out_n_accepted, void *stream);

/*
 * spec_verify_ex — spec_verify plus optional observability outputs.
 *   out_row_max     [B, 2K+1] float or NULL: max logit of each row
 *   out_row_sumexp  [B, 2K+1] float or NULL: S = sum_v exp((z_v - max)/T)
 *                   (NaN when T == 0).  Row order: target rows 0..K, then
 *                   draft rows 0..K-1 (draft rows are NaN when T == 0).
 *   stats           spec_stats_t* in device memory or NULL (accumulated)
 */
int spec_verify_ex(const void *target_logits, const void *draft_logits,
                   const int32_t *draft_tokens, int B, int K, int V, int dtype,
                   float temperature, uint64_t seed, int32_t *out_tokens,
                   int32_t *out_n_accepted, float *out_row_max,
                   float *out_row_sumexp, spec_stats_t *stats, void *stream);

/*
 * spec_verify_host — spec_verify on HOST buffers, end to end and synchronous:
 * copies the inputs to a library-owned device staging area (grow-only, per
 * device and stream), verifies, copies the outputs back and waits.  Page-
 * locked host buffers give the fastest copies.  Returns SPEC_OK, an argument
 * error, or the device status of this call (as spec_get_status).
 */
int spec_verify_host(const void *target_logits, const void *draft_logits,
                     const int32_t *draft_tokens, int B, int K, int V, int dtype,
                     float temperature, uint64_t seed, int32_t *out_tokens,
                     int32_t *out_n_accepted, void *stream);

/*
 * spec_verify_noalloc — spec_verify for callers that cannot allocate device
 * memory while they run: a serving engine that hands nearly all of HBM to
 * its own memory pool at start-up, or a latency-critical loop that cannot
 * afford cudaMalloc/cudaFree (cudaFree can synchronise the whole device).
 * The pages describe no such interface; it exists for integration only.
 *
 * Same arguments, outputs and results as spec_verify (temperature > 0 and
 * T == 0 alike), but the scratch space comes from a fixed array compiled into
 * the library (a status word, the streaming kernel's item counters, which
 * every call leaves at zero, and 8 MiB of row partials), which every GPU
 * that loads the library keeps until the process exits.  Nothing is
 * allocated by the call.
 *
 *   - Size limit: B * (K+1) * ceil(V * element_size / 16384) <= 65536
 *     (e.g. B = 64, K = 5, V = 128256 bf16 uses 6144).  Larger calls return
 *     SPEC_ERR_ARG with an explanation and launch nothing.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call shares the one array: two calls that overlap on the GPU
 *     (different streams, or different host threads) race and corrupt each
 *     other's results.  Serialise them.
 *   - Errors found on the device show in the outputs: a draft token outside
 *     [0, V) marks its sequence (n_accepted = -1, tokens -1); a bounded wait
 *     that ran out marks every sequence of the call, and of every later
 *     call, until spec_noalloc_get_status reads and clears the array's
 *     status word (spec_get_status does not read it).
 *   - After a device reset (cudaDeviceReset) call spec_shutdown before the
 *     next call: it forgets the array's cached device addresses.
 */
int spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, int B, int K, int V, int dtype,
                        float temperature, uint64_t seed, int32_t *out_tokens,
                        int32_t *out_n_accepted, void *stream);

/*
 * spec_noalloc_get_status — spec_get_status for the status word of
 * spec_verify_noalloc's fixed array: waits for `stream` (the stream the calls
 * ran on), then returns and clears the first device-side error recorded by
 * those calls (SPEC_OK, SPEC_ERR_TOKEN_RANGE or SPEC_ERR_TIMEOUT).
 * Allocates nothing; like the first spec_verify_noalloc call on a device,
 * its first call looks up the array's device address.
 */
int spec_noalloc_get_status(void *stream);

/*
 * spec_verify_tree_greedy — greedy verification of a draft tree
 * ([Infra53] §3: every node sees only its ancestors, one path is
 * committed; [Anhtu] §"Token tree": the deepest accepted branch is the
 * output).  Row n of target_logits is the target's distribution after node
 * n.  Node c >= 1 is accepted iff its parent is accepted and
 * node_tokens[b, c] == argmax(target_logits[b, parent[c], :]) (lowest index
 * on ties); node 0 (the root, already committed) is always accepted.  The
 * deepest accepted node d* (lowest index among equals) is committed.
 *
 *   target_logits  [B, N, V], dtype
 *   parent         [N] int32 (device): parent[0] = -1, 0 <= parent[c] < c
 *   node_tokens    [B, N] int32; entry 0 is ignored
 *   B >= 0, 1 <= N <= SPEC_MAX_TREE_NODES, V >= 1
 *   max_depth      D = spec_tree_max_depth(parent) (from a host copy)
 *   out_path       [B, D+1] int32: tokens of the committed path (root
 *                  excluded), then the bonus argmax(row d*), then -1 padding
 *   out_len        [B] int32: depth(d*) + 1, or -1 on a device error
 * A parent[] that is not a tree, or deeper than max_depth, is reported as
 * SPEC_ERR_PARENT by spec_get_status and sets every out_len to -1.
 */
int spec_verify_tree_greedy(const void *target_logits, const int32_t *parent,
                            const int32_t *node_tokens, int B, int N, int V,
                            int dtype, int max_depth, int32_t *out_path,
                            int32_t *out_len, void *stream);

/*
 * spec_verify_tree — stochastic verification of a draft tree at temperature
 * T > 0 (T == 0 is greedy matching, as spec_verify_tree_greedy).  The pages
 * give the chain rule ([Oscine] §"验收标准的精确数学", §"拒绝之后怎么办？——
 * 残差分布") and warn that verifying a tree does not by itself keep the
 * output lossless ([Infra53] §9); the rule for several children of a node is
 * not given, and this reading is the lossless extension of the chain rule:
 * the children of a node are candidates drawn independently from the
 * draft's distribution q at that node, tried in index order.  With r the
 * current target distribution at the node (r = p at first), candidate x is
 * accepted iff u < r(x)/q(x); a reject replaces r by norm(max(0, r - q)).
 * An accepted candidate becomes the current node; a node whose candidates
 * are all rejected emits a token drawn from r; an accepted node without
 * children emits a bonus token drawn from its p.  Only one path is
 * committed ([Infra53] §3).  Uniforms: the test of child c uses counter
 * (b, c - 1, slot 0), the draw at node u uses (b, u, slot 1); a chain-shaped
 * tree (parent[c] = c - 1) therefore gives exactly spec_verify's result.
 *
 *   target_logits  [B, N, V], dtype: row u = target distribution at node u
 *   draft_logits   [B, N, V], dtype: row u = draft distribution at node u,
 *                  from which u's children were drawn (rows of nodes
 *                  without children are not read)
 *   parent         [N] int32 (device): parent[0] = -1, 0 <= parent[c] < c
 *   node_tokens    [B, N] int32; entry 0 is ignored
 *   B >= 0, 1 <= N <= SPEC_MAX_TREE_NODES, V >= 1, T >= 0, seed as spec_verify
 *   max_depth      D = spec_tree_max_depth(parent) (from a host copy)
 *   out_path       [B, D+1] int32: tokens of the accepted path (root
 *                  excluded), then the emitted token, then -1 padding
 *   out_len        [B] int32: accepted + 1, or -1 on a device error
 * A token outside [0, V) is reported as SPEC_ERR_TOKEN_RANGE, a parent[]
 * that is not a tree of depth <= max_depth as SPEC_ERR_PARENT (both by
 * spec_get_status); the sequence's outputs are -1.
 */
int spec_verify_tree(const void *target_logits, const void *draft_logits,
                     const int32_t *parent, const int32_t *node_tokens, int B, int N,
                     int V, int dtype, float temperature, uint64_t seed, int max_depth,
                     int32_t *out_path, int32_t *out_len, void *stream);

/*
 * spec_verify_trees_greedy, spec_verify_trees — the same two verifications
 * with one tree per sequence, as a dynamic tree budget builds them
 * ([Infra53] §5.1: EAGLE-2 grows a different tree for each context; see
 * spec_eagle2_rerank, whose listing is such a tree):
 *   parents  [B, N] int32 (device): row b is sequence b's tree (parent[0] =
 *            -1, parent[c] < c, depth <= max_depth, checked on the device)
 * Everything else as spec_verify_tree_greedy / spec_verify_tree.  With one
 * tree per sequence the stochastic form streams every node's draft row (which
 * nodes have children differs between sequences), so it reads B*2N rows.
 */
int spec_verify_trees_greedy(const void *target_logits, const int32_t *parents,
                             const int32_t *node_tokens, int B, int N, int V, int dtype,
                             int max_depth, int32_t *out_path, int32_t *out_len, void *stream);
int spec_verify_trees(const void *target_logits, const void *draft_logits, const int32_t *parents,
                      const int32_t *node_tokens, int B, int N, int V, int dtype, float temperature,
                      uint64_t seed, int max_depth, int32_t *out_path, int32_t *out_len, void *stream);

/*
 * spec_tree_max_depth — HOST helper: the largest node depth of parent[]
 * (HOST pointer), or -SPEC_ERR_PARENT if parent[] is not a tree
 * ([Infra53] §3.2: position IDs follow tree depth).
 */
int spec_tree_max_depth(const int32_t *parent_host, int N);

/*
 * spec_tree_mask — tree-attention mask and depth position IDs of B trees
 * ([Infra53] §3.1–§3.2 and the example of §8: node n sees exactly its
 * ancestors and itself; its position ID is its depth).
 *   parent     [B, N] int32 (device), each row a tree as above
 *   out_mask   [B, N, W] uint32 with W = ceil(N / 32): bit (a mod 32) of
 *              word a / 32 of row n is set iff a is an ancestor-or-self of n
 *   out_depth  [B, N] int32
 * A malformed tree is reported by spec_get_status (SPEC_ERR_PARENT) and its
 * rows are zeroed with depth -1.
 */
int spec_tree_mask(const int32_t *parent, int B, int N, uint32_t *out_mask,
                   int32_t *out_depth, void *stream);

/*
 * spec_verify_points — chain verification of drafts from a deterministic
 * drafter, such as spec_ngram_propose, which proposes tokens but no
 * distribution ([Glukhov] §"Спекулятивное декодирование на n-граммах").
 * Reading taken: the chain rule of spec_verify with q_i the point mass at
 * x_i: x_i is accepted iff u < p_i(x_i); at the first reject j the token is
 * drawn from max(0, p_j - q_j), i.e. p_j without x_j; if all k drafts are
 * accepted the bonus comes from p_k.  Equal to spec_verify with draft logits
 * that are 0 at x_i and -inf elsewhere, without reading any draft rows.
 *   target_logits [B, K+1, V]; draft_tokens [B, K] (device)
 *   draft_counts  [B] int32 (device) or NULL: sequence b verifies its first
 *                 k = draft_counts[b] drafts (0 <= k <= K; the rest are not
 *                 read, e.g. -1 from spec_ngram_propose) and draws its bonus
 *                 from p_k (target row k)
 *   out_tokens [B, K+1]: accepted drafts, the new token, then -1;
 *   out_n_accepted [B].  T = 0 is greedy matching of the k drafts.
 * Uniforms, errors and limits as spec_verify; a count outside [0, K] is
 * reported like an out-of-range token.
 */
int spec_verify_points(const void *target_logits, const int32_t *draft_tokens,
                       const int32_t *draft_counts, int B, int K, int V, int dtype,
                       float temperature, uint64_t seed, int32_t *out_tokens,
                       int32_t *out_n_accepted, void *stream);

/*
 * spec_ngram_propose — n-gram (prompt-lookup) drafting: for each of B
 * contexts, the up to K tokens that followed an earlier occurrence of the
 * context's own last n tokens ([Glukhov] §"Спекулятивное декодирование на
 * n-граммах"; the window n_max is [Anhtu] §"Bật trong production"'s
 * prompt_lookup_max, min_hits [Glukhov] §"Настройка параметров"'s min-hits).
 * The pages leave the choice among several matches open; this reading is
 * taken: the longest n in [n_min, n_max] whose suffix t[len-n .. len-1]
 * occurred at least min_hits times at earlier starts j (j + n <= len - 1,
 * so at least one token follows the occurrence) wins, and of those
 * occurrences the most recent (largest j); the proposal is
 * t[j+n .. j+n+count-1] with count = min(K, len - j - n).
 *   tokens     [B, L] int32 (device): row b holds the context of sequence b
 *              in its first lengths[b] entries; the rest is not read
 *   lengths    [B] int32 (device), 0 <= lengths[b] <= L
 *   n_min, n_max  1 <= n_min <= n_max <= SPEC_MAX_NGRAM
 *   min_hits   >= 1 (1: any earlier occurrence)
 *   K          0 <= K <= SPEC_MAX_DRAFTS
 *   out_draft  [B, K] int32 (device): the proposal, then -1
 *   out_count  [B] int32 (device): tokens proposed (0: no match)
 * Token values are compared as plain integers and never range-checked.  A
 * lengths[b] outside [0, L] sets out_count[b] = -1 and its draft row to -1,
 * and spec_get_status then returns SPEC_ERR_ARG.  Output is bit-exact and
 * deterministic (a pure function of the inputs).
 * Launch geometry: G CTAs share each context's end positions: one round of
 * loads each (4096 positions) when the batch then fits in about one wave of
 * resident CTAs (up to 1.25 waves), else as many as one wave holds.  They
 * combine their partials through one thread-block cluster when G <= 8 and
 * through global memory otherwise.  The environment variable
 * SPEC_NGRAM_CTAS, read at each call, sets G instead (any G >= 1 gives the
 * same outputs).
 */
int spec_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B, int L, int n_min,
                       int n_max, int min_hits, int K, int32_t *out_draft, int32_t *out_count,
                       void *stream);

/*
 * spec_topk — the k most probable tokens of each of R rows and their
 * probabilities under softmax(z / T): the confidences of the EAGLE-2 tree
 * budget ([Infra53] §5.1-§5.2: the draft's confidence decides where the
 * node budget goes).
 *   logits      [R, V] SPEC_F32 or SPEC_BF16 (device)
 *   1 <= k <= min(V, SPEC_MAX_TOPK), T > 0
 *   out_tokens  [R, k] int32 (device): by decreasing logit, ties to the
 *               lower index
 *   out_prob    [R, k] float (device): softmax(z / T) of those tokens
 * Rows must hold one finite logit (-inf entries allowed).
 * Launch geometry: each row is split over a cluster of G CTAs of 512
 * threads (G a power of two up to 8, about one wave of 1.5 CTAs per SM, each
 * slice at least 32 KB; G = 1 when the rows alone fill that wave); the
 * environment variable SPEC_TOPK_CLUSTER, read at each call, sets G instead
 * (rounded down to a power of two; any G gives the same outputs).  No other
 * environment variable changes this library's launches.
 */
int spec_topk(const void *logits, int R, int V, int dtype, float temperature, int k,
              int32_t *out_tokens, float *out_prob, void *stream);

/*
 * spec_eagle2_expand — one expansion step of the EAGLE-2 tree budget for B
 * trees ([Infra53] §5.2: a node's value is the product of the confidences on
 * its path; the expansion phase grows the few best nodes).  Reading taken:
 * each frontier node offers its k most probable tokens (spec_topk of the
 * draft's row at that node) as candidates; a candidate's value is its
 * parent's value times its probability; the k_next candidates of highest
 * value (ties to the lower node id) become the next frontier.
 *   draft_logits  [B, F, V] (device): the draft's logits at the frontier
 *   frontier      [B, F] int32 (device): node ids in [0, offset)
 *   node_tokens, node_values, node_parents  [B, cap] int32 / float / int32
 *                 (device, caller-owned tree state): node 0 is the root (the
 *                 caller sets value 1, parent -1 and its token); the step
 *                 writes the F * k candidates to nodes offset + f * k + j
 *                 (j = 0..k-1 in decreasing probability), offset >= 1,
 *                 offset + F * k <= cap, F * k <= SPEC_EAGLE_MAX_CANDIDATES
 *   out_frontier  [B, k_next] int32 (device): node ids, best first
 *                 (0 <= k_next <= F * k)
 * A frontier id outside [0, offset) makes spec_get_status return
 * SPEC_ERR_PARENT and that tree's out_frontier -1.  Two launches.
 */
int spec_eagle2_expand(const void *draft_logits, const int32_t *frontier, int B, int F, int V,
                       int dtype, float temperature, int k, int32_t *node_tokens,
                       float *node_values, int32_t *node_parents, int cap, int offset, int k_next,
                       int32_t *out_frontier, void *stream);

/*
 * spec_eagle2_rerank — the rerank phase ([Infra53] §5.2: keep the best
 * nodes of all for verification).  For each of B trees of M nodes (arrays
 * [B, M] as written by spec_eagle2_expand; parent[0] = -1, parent[c] < c):
 * keeps the root and the m other nodes of highest value, ties to the
 * smaller depth, then the lower id (depth < 256).  A child's value never
 * exceeds its parent's, so the kept set holds every ancestor of a kept node.
 *   out_parent  [B, m + 1] int32 (device): parents as list positions (-1
 *               for the root); the list is the root, then the kept nodes by
 *               depth, then by rank, so parent[c] < c (ready for
 *               spec_tree_mask and the tree verification)
 *   out_tokens  [B, m + 1] int32: their tokens; out_index [B, m + 1]: node ids
 * 1 <= M <= SPEC_EAGLE_MAX_NODES, 0 <= m <= M - 1.  A malformed tree, or a
 * kept node whose parent was dropped, makes spec_get_status return
 * SPEC_ERR_PARENT and that tree's outputs -1.
 */
int spec_eagle2_rerank(const float *node_values, const int32_t *node_parents,
                       const int32_t *node_tokens, int B, int M, int m, int32_t *out_parent,
                       int32_t *out_tokens, int32_t *out_index, void *stream);

/*
 * spec_get_status — waits for `stream`, then returns (and clears) the first
 * device-side error recorded by calls on it: SPEC_OK, SPEC_ERR_TOKEN_RANGE,
 * SPEC_ERR_PARENT, SPEC_ERR_TIMEOUT, SPEC_ERR_ARG (a lengths[] entry of
 * spec_ngram_propose out of range), or SPEC_ERR_CUDA for an asynchronous
 * CUDA error.  While a SPEC_ERR_TIMEOUT is recorded and not yet read, every
 * verification on the stream (chains, point-mass drafts, trees) writes -1
 * for its outputs (n_accepted or length -1, tokens -1) instead of values
 * drawn from statistics a stopped wait may have left incomplete.
 */
int spec_get_status(void *stream);

/*
 * spec_arm_rows_event — measurement hook.  The next verification call that
 * launches (any spec_verify* entry point: chains, point-mass drafts, trees)
 * made by the calling host thread records `event`
 * (a cudaEvent_t created by the caller, passed as void*) on its stream right
 * after launching its streaming kernel (the row statistics) and before its
 * decision kernel; the hook is then disarmed.  An event the caller records
 * just before that call and this one bracket the streaming kernel alone.
 * The decision kernel of that call then starts only after the event, so
 * calls timed this way are for measurement, not for the fastest throughput.
 * Always returns SPEC_OK.
 */
int spec_arm_rows_event(void *event);

/*
 * spec_arm_timer — measurement hook that leaves the stream untouched: the
 * next verification call (any spec_verify* entry point) or top-k launch
 * (spec_topk, or the top-k of spec_eagle2_expand) made by the calling host
 * thread records global-timer stamps (%globaltimer, ns) into `stamps`, three
 * unsigned 64-bit words in device memory that the caller has set to
 * (UINT64_MAX, 0, 0).  Verification: [0] the earliest start of a streaming
 * CTA (after its wait on the preceding work), [1] the latest end of one, [2]
 * the latest output written by the decision kernel.  Top-k: [0] the earliest
 * CTA start (after the wait), [1] the latest CTA end, [2] the latest row
 * written.  No event or other operation is put between the launches, so
 * calls made back to back still chain by programmatic dependent launch, and
 * [1] - [0] is the kernel's time as it runs there.  The hook is then
 * disarmed.  Always returns SPEC_OK.
 */
int spec_arm_timer(unsigned long long *stamps);

/*
 * spec_selftest_wait — diagnostic of the bounded waits every kernel uses on
 * its barriers: one thread waits on a barrier that nothing completes; the
 * wait gives up after one second of global time or 2^17 polls, whichever
 * comes first (about half a second on GB300), the kernel records a
 * timeout and returns.  The next spec_get_status on `stream` then returns
 * SPEC_ERR_TIMEOUT, and the stream stays usable.  Returns SPEC_OK once
 * launched.
 */
int spec_selftest_wait(void *stream);

/*
 * spec_debug_fail_launch — fault injection for tests of the error paths: the
 * n-th kernel launch from now (counting every launch of this library, n >=
 * 1) fails with a launch error instead of launching; the call that made it
 * returns SPEC_ERR_CUDA and leaves the stream's workspace ready for the next
 * call.  n = 0 switches it off.  No GPU fault is involved.
 */
int spec_debug_fail_launch(int n);

/*
 * spec_debug_noalloc_status — test hook of spec_verify_noalloc's error path:
 * ORs the device status bits `bits` (1: token out of range, 4: a wait ran
 * out) into the status word of its fixed array, as a kernel would, so that
 * a test can check the outputs and spec_noalloc_get_status without faulting
 * or stalling a GPU.  Synchronous; allocates nothing.
 */
int spec_debug_noalloc_status(int bits);

/* Static, human-readable name of a status code. */
const char *spec_error_string(int status);

/* Detail of the last error returned on the calling host thread. */
const char *spec_last_error_message(void);

/* Frees every workspace and staging buffer the library holds.  No call may
 * be in flight. */
void spec_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
