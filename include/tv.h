/*
 * tv.h -- C ABI of the GB300 tree verify round.
 *
 * One verify round of speculative decoding [Drafters and tree verify, §The
 * round]: (2) one forward pass scores every node of a draft tree of at most 32
 * nodes against the KV cache, (3) a walk accepts a root path, (4) the commit
 * keeps only the accepted path's KV rows.  Every entry point is asynchronous
 * on the given CUDA stream and runs hand-written sm_103a kernels; there is no
 * CPU fallback.
 *
 * Conventions shared by all entry points
 * --------------------------------------
 * - bf16 values are passed as uint16_t bit patterns (tv_bf16).
 * - "device" pointers point to memory the GPU can read/write (cudaMalloc'd or
 *   torch CUDA tensors); "host" values are plain C values read during the call.
 * - The caller owns every buffer.  The library allocates nothing: scratch
 *   space is the caller's workspace, sized by tv_workspace_size().
 * - A draft tree is a parent array in parent-before-child order: parent[0] = -1
 *   (the root, the round's anchor token whose K/V this verify computes) and
 *   0 <= parent[i] < i, with no two siblings carrying the same token
 *   [Algorithm and correctness contract, §Target position and batching].
 *   Depth-first pre-order [Drafters and tree verify, §Tree verify through
 *   recurrent layers] is one such order; any parent-before-child order works.
 * - Row i of a tree scores node i's children: it processes node i's token at
 *   position ctx + depth(i) and attends to the cached context plus the
 *   root-to-i path, i included.  Siblings therefore share the parent's row
 *   [Algorithm and correctness contract, §Target position and batching].
 * - Several requests may share one pass (joint verify [Exactness, §Parallel
 *   requests]): their rows are concatenated in request order, at most 32 rows
 *   in all; request r owns rows row_off(r) .. row_off(r) + n_r - 1 of every
 *   per-row array, where row_off(r) = n_0 + ... + n_{r-1}.  Each request has
 *   its own cache and sees only its own cache and its own ancestors.
 *
 * Errors
 * ------
 * Every entry point returns TV_OK (0) or a negative TV_E_* code.  Checks that
 * need only host values happen before anything is launched; nothing is
 * launched when one fails.  Checks that need device data (the tree arrays, the
 * uniforms) run in the kernels, which then write the code into *dev_status.
 * dev_status is sticky: kernels only ever change it from 0 to a code, and every
 * kernel of every entry point does nothing while it is non-zero.  So a caller
 * can chain verify -> accept -> commit with one status word, zeroed once per
 * round, and read it after the round; a commit never runs on a bad path.
 * Device waits are bounded: a wait that gives up writes TV_E_TIMEOUT.
 */
#ifndef TV_H
#define TV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* the library is built with hidden visibility; these are its only exports */
#if defined(__GNUC__)
#define TV_API __attribute__((visibility("default")))
#else
#define TV_API
#endif

#define TV_OK              0
#define TV_E_ARG          -1   /* a null pointer, a bad size or a bad dims field        */
#define TV_E_ORDER        -2   /* parent[0] != -1 or parent[i] not in [0, i)            */
#define TV_E_DUP_SIBLING  -3   /* two children of one node carry the same token         */
#define TV_E_TOKEN        -4   /* a token id outside [0, vocab)                         */
#define TV_E_CAPACITY     -5   /* ctx_len + n > capacity                                */
#define TV_E_ROWS         -6   /* a tree outside 1..32 nodes, or more than 32 rows total */
#define TV_E_UNIFORM      -7   /* a uniform that is not finite or not in [0, 1)         */
#define TV_E_TEMP         -8   /* temperature not finite or <= 0                        */
#define TV_E_WORKSPACE    -9   /* workspace null or smaller than tv_workspace_size()    */
#define TV_E_CUDA        -10   /* a CUDA runtime call failed                            */
#define TV_E_UNSUPPORTED -11   /* a shape these kernels do not handle (see tv_dims)     */
#define TV_E_TIMEOUT     -12   /* a bounded device wait gave up                         */
#define TV_E_PATH        -13   /* commit: accept_len or a path entry out of range       */
#define TV_E_CHAIN       -14   /* single-path sampling on a tree that is not a chain    */
#define TV_E_PROPOSAL    -15   /* a proposal row not finite, negative, off unit mass, or
                                  zero at its draft                                     */

typedef uint16_t tv_bf16;

/* Shapes of the layer.  Supported: head_dim 64 or 128; hidden and
 * n_q_heads*head_dim multiples of 64; n_q_heads a multiple of n_kv_heads;
 * (n_q_heads / n_kv_heads) * (rows of one request) <= 160; vocab >= 2. */
typedef struct tv_dims {
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, vocab;
  float rope_theta;   /* RoPE base (rotate-half pairs (d, d + head_dim/2)) */
  float rms_eps;      /* RMSNorm epsilon                                    */
} tv_dims;

/* The layer + head, all device pointers to bf16, caller-owned:
 *   embed   [vocab][hidden]            token embedding
 *   ln1     [hidden]                   RMSNorm gain before the projections
 *   wqkv    [(Hq + 2 Hkv) D][hidden]   rows: the Q heads, then K heads, then V heads
 *   wo      [hidden][Hq D]             output projection
 *   ln_f    [hidden]                   final RMSNorm gain
 *   lm_head [vocab][hidden]            output head
 * packed = 0: wqkv, wo and lm_head are row-major as above.  packed = 1: each
 * of the three is the tile-packed copy tv_pack_weight makes of that matrix
 * (the same numbers; the GEMMs then read every 16 KB tile from one contiguous
 * stretch of memory, which streams faster).  Every other pointer is row-major
 * either way.                                                                  */
typedef struct tv_model {
  const tv_bf16 *embed, *ln1, *wqkv, *wo, *ln_f, *lm_head;
  tv_dims dims;
  int32_t packed;
} tv_model;

/*
 * The tile-packed layout of a bf16 weight W [rows][cols] (cols a multiple of
 * 64): the rows are padded with zeros to a multiple of 128, cut into tiles of
 * 128 rows x 64 columns, and tile (i, j) (rows 128 i .., columns 64 j ..) is
 * stored row-major at element offset (i * (cols / 64) + j) * 8192.
 *
 * tv_packed_weight_bytes: host-only; writes the packed size in bytes
 * (ceil(rows / 128) * 128 * cols * 2).  TV_E_ARG on rows < 1 or cols not a
 * positive multiple of 64.
 * tv_pack_weight: device W (row-major, 16-byte aligned) -> device packed
 * (16-byte aligned, tv_packed_weight_bytes bytes, caller-owned, not
 * overlapping W), enqueued on `stream`; meant to run once when the weights are
 * loaded.  TV_E_ARG as above or on null / unaligned pointers, TV_E_CUDA if
 * the launch fails.
 */
TV_API int tv_packed_weight_bytes(int32_t rows, int32_t cols, size_t *bytes);
TV_API int tv_pack_weight(const tv_bf16 *w, int32_t rows, int32_t cols, tv_bf16 *packed, void *stream);

/* One request's KV cache, device pointers to bf16, layout [Hkv][capacity][D].
 * Slots [0, ctx_len) hold the cached context.  ctx_len and capacity are host
 * values; the caller advances ctx_len after a commit (new_ctx). */
typedef struct tv_kv {
  tv_bf16 *k, *v;
  int32_t ctx_len, capacity;
} tv_kv;

/* One request's draft tree: device int32 arrays of n entries; n is a host value. */
typedef struct tv_tree {
  const int32_t *parent, *token;
  int32_t n;
} tv_tree;

/*
 * Bytes of workspace that tv_verify_tree and tv_accept_residual need for any
 * round of up to max_rows rows (<= 32) whose requests have ctx_len <= max_ctx.
 * Host-only; writes *bytes.  Returns TV_E_ARG / TV_E_UNSUPPORTED on bad dims.
 */
TV_API int tv_workspace_size(const tv_dims *dims, int max_rows, int max_ctx, size_t *bytes);

/*
 * The verify pass [Drafters and tree verify, §The round, step 2; §Tree verify
 * through recurrent layers]: one forward pass over every row of n_req trees.
 *
 *   model        host struct of device weight pointers
 *   kv           host array [n_req]; verify writes row i's K/V into slot
 *                ctx_len + i of its request's cache ("the cache holds every node
 *                at its depth-first slot"); slots below ctx_len are only read
 *   trees        host array [n_req]
 *   logits       device fp32 [total_rows][vocab] -- the head's fp32 logits
 *                [Exactness, §The one exception: near ties]
 *   argmax       device int32 [total_rows] -- per row the index of the largest
 *                logit, the lowest index among equal maxima
 *   top2_gap     device fp32 [total_rows] -- largest minus second-largest logit
 *                (0 when the maximum is attained twice)
 *   attn_out     device bf16 [total_rows][Hq*D] or NULL -- attention output
 *   workspace    device, >= tv_workspace_size(dims, total_rows, max ctx_len)
 *   dev_status   device int32, sticky (see Errors)
 *   stream       cudaStream_t (NULL = legacy default stream)
 *
 * Host checks: TV_E_ARG, TV_E_ROWS, TV_E_CAPACITY, TV_E_WORKSPACE,
 * TV_E_UNSUPPORTED.  Device checks (-> *dev_status): TV_E_ORDER,
 * TV_E_DUP_SIBLING, TV_E_TOKEN.  Every row's logits use one reduction order,
 * fixed by the weight shapes and never by the row count, so a row's results do
 * not depend on the other rows in the pass [Exactness, §Parallel requests].
 */
TV_API int tv_verify_tree(const tv_model *model, const tv_kv *kv, const tv_tree *trees, int n_req,
                   float *logits, int32_t *argmax, float *top2_gap, tv_bf16 *attn_out,
                   void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Greedy accept [Drafters and tree verify, §The round, step 3]: walk down from
 * the root; at each node take the model's token (argmax of its row); move to
 * the child that carries it; stop where no child does; keep the model's token
 * at the stopping node too, so a round yields at least one token.
 *
 *   trees        host array [n_req]
 *   argmax       device int32 [total_rows] (from tv_verify_tree)
 *   path         device int32 [total_rows]: request r's accepted node indices,
 *                root first, at path[row_off(r) .. row_off(r) + a_r]
 *   accept_len   device int32 [n_req]: a_r = accepted non-root nodes
 *   out_tokens   device int32 [total_rows]: the a_r accepted drafts then the
 *                stopping node's token, a_r + 1 tokens at row_off(r)
 *   dev_status   device int32, sticky.  Device checks: TV_E_ORDER,
 *                TV_E_DUP_SIBLING.
 */
TV_API int tv_accept_greedy(const tv_tree *trees, int n_req, const int32_t *argmax,
                     int32_t *path, int32_t *accept_len, int32_t *out_tokens,
                     int32_t *dev_status, void *stream);

/*
 * Deterministic-candidate residual sampling [Algorithm and correctness
 * contract, §Deterministic tree candidates and residual verification]: at the
 * current node r := p = softmax(logits_row / temperature); its children are
 * tried in increasing node index: accept candidate x iff u < r(x); on
 * rejection remove x from r and renormalise; on acceptance follow that child.
 * If every child fails, draw one token from the residual r, emit it, end.
 * At a leaf the round ends; if bonus_at_leaf, one draw from p is emitted there
 * (the target's own token at the stopping point, as the greedy walk keeps it).
 * A draw y from r is the smallest y with sum_{j<=y} r(j) > u * sum(r).
 *
 *   logits       device fp32 [total_rows][vocab] (from tv_verify_tree)
 *   uniforms     device fp32 [total_rows]: request r consumes
 *                uniforms[row_off(r) ..] in order, one per candidate test and
 *                one for the final draw (at most n_r draws)
 *   path, accept_len  as tv_accept_greedy
 *   out_tokens   device int32 [total_rows]; out_count device int32 [n_req]
 *                holds how many tokens request r emitted (a_r or a_r + 1)
 *   workspace    device, >= tv_workspace_size(dims with this vocab, total_rows, 0)
 * Host checks: TV_E_TEMP, TV_E_ARG, TV_E_ROWS, TV_E_WORKSPACE.  Device checks:
 * TV_E_ORDER, TV_E_DUP_SIBLING, TV_E_TOKEN, TV_E_UNIFORM.
 */
TV_API int tv_accept_residual(const tv_tree *trees, int n_req, const float *logits, int32_t vocab,
                       float temperature, const float *uniforms, int bonus_at_leaf,
                       int32_t *path, int32_t *accept_len, int32_t *out_tokens, int32_t *out_count,
                       int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * tv_accept_residual without a workspace.  The pages have no counterpart: this
 * is for callers that cannot provide device memory -- a plugin step inside
 * another framework's executor that may not call cudaMalloc, a real-time loop
 * with a no-allocation rule, a caller holding only a stream and the round's
 * buffers.  Same walk, same kernels and same results as tv_accept_residual; the
 * per-row softmax statistics live instead in a 272 KB array inside the
 * library's device image (one per GPU, held until the process exits), so:
 *   - vocab may be at most 262144 (TV_E_UNSUPPORTED above that);
 *   - every call looks up that array's address in the context current on
 *     the calling thread (cudaGetSymbolAddress, a host-side lookup; nothing
 *     is cached, so another context or a reset device never sees a stale
 *     address); the first call in a context also loads the library's device
 *     image there -- make it before any stream capture;
 *   - all calls on a device share the array: calls whose kernels overlap on the
 *     GPU race; order them on one stream.
 * Nothing is allocated.  Arguments and errors as tv_accept_residual.
 */
TV_API int tv_accept_residual_noalloc(const tv_tree *trees, int n_req, const float *logits, int32_t vocab,
                                      float temperature, const float *uniforms, int bonus_at_leaf,
                                      int32_t *path, int32_t *accept_len, int32_t *out_tokens,
                                      int32_t *out_count, int32_t *dev_status, void *stream);

/*
 * KV commit [Drafters and tree verify, §The round, step 4; §Tree verify through
 * recurrent layers, last paragraph]: keep the accepted path's KV rows and drop
 * the rest -- for d = 0..a_r, copy slot ctx_len + path[d] to slot ctx_len + d,
 * every KV head, K and V.  All source rows are read before any row is written
 * (a target slot can be an earlier step's source).
 *
 *   kv           host array [n_req] (the same caches verify wrote into)
 *   trees        host array [n_req] (only n is read, for the row offsets)
 *   path, accept_len  device, from an accept walk
 *   committed_src device int32 [total_rows]: slot ctx_len + path[d] for
 *                d = 0..a_r at row_off(r)
 *   new_ctx      device int32 [n_req]: ctx_len + a_r + 1
 * Host checks: TV_E_ARG, TV_E_ROWS.  Device checks: TV_E_PATH.
 */
TV_API int tv_commit_kv(const tv_kv *kv, const tv_dims *dims, const tv_tree *trees, int n_req,
                 const int32_t *path, const int32_t *accept_len,
                 int32_t *committed_src, int32_t *new_ctx, int32_t *dev_status, void *stream);

/*
 * The greedy walk and the KV commit in one launch [Drafters and tree verify,
 * §The round, steps 3 and 4]: the outputs of tv_accept_greedy followed by
 * tv_commit_kv on the same arguments -- path, accept_len, out_tokens,
 * committed_src, new_ctx and the cache rows -- with one kernel instead of two.
 * The path comes from the walk, so TV_E_PATH cannot arise.
 *
 *   kv, dims, trees  as tv_commit_kv (trees: the device parent/token arrays
 *                    are read, as by tv_accept_greedy)
 *   argmax           device int32 [total_rows], from tv_verify_tree
 *   the rest         as those two calls
 * Host checks: TV_E_ARG, TV_E_ROWS, TV_E_UNSUPPORTED.  Device checks:
 * TV_E_ORDER, TV_E_DUP_SIBLING.
 */
TV_API int tv_accept_greedy_commit(const tv_kv *kv, const tv_dims *dims, const tv_tree *trees, int n_req,
                                   const int32_t *argmax, int32_t *path, int32_t *accept_len, int32_t *out_tokens,
                                   int32_t *committed_src, int32_t *new_ctx, int32_t *dev_status, void *stream);

/*
 * Sampled variants [Exactness, §Sampling; Drafters and tree verify,
 * §Sampling; Algorithm and correctness contract, §Single-path sampling].
 * They read the verify's fp32 logits (or the output of tv_sample_filter with
 * temperature 1) and need a workspace of tv_sample_workspace_size() bytes.
 */

/* Bytes of workspace the sampled entry points need for up to max_rows rows
 * (<= 32) of this vocabulary.  Host-only. */
TV_API int tv_sample_workspace_size(int32_t vocab, int max_rows, size_t *bytes);

/*
 * Sampling filters through one function [Exactness, §Sampling, second
 * paragraph]: filtered[row][y] = logits[row][y] / temperature for the tokens
 * the filters keep and -inf for the rest, so that softmax(filtered) is the
 * filtered, renormalised distribution and every sampled walk can run on it
 * with temperature 1 (drafted rows and plain rows see the same filters).
 * Applied in this order, each on the distribution the previous ones left:
 *   top_k (0 = off)  keep the tokens whose logit is at least the k-th largest
 *                    (tokens tied with it are all kept);
 *   top_p (1 = off)  keep the fewest largest-probability tokens whose mass
 *                    reaches top_p (ties at the boundary all kept);
 *   min_p (0 = off)  keep the tokens with p >= min_p * max p.
 * The k-th largest logit and the top-p boundary are found exactly (integer
 * histograms over the logits' bits; probability masses in units of 2^-40),
 * so the result does not depend on the run.  Each row is handled by a
 * cluster of 8 CTAs holding the row in shared memory, hence the vocabulary
 * limit.
 *
 *   logits    device fp32 [rows][vocab];  filtered  device fp32 [rows][vocab]
 *             (may not alias logits)
 * Host checks: TV_E_ARG (null pointers, rows outside 1..32, vocab < 2,
 * top_k < 0, top_p outside (0, 1], min_p outside [0, 1)), TV_E_TEMP,
 * TV_E_UNSUPPORTED (vocab > 262144).
 */
TV_API int tv_sample_filter(const float *logits, float *filtered, int rows, int32_t vocab, float temperature,
                            int32_t top_k, float top_p, float min_p, int32_t *dev_status, void *stream);

/*
 * Single-draw sampled verify [Exactness, §Sampling, first paragraph; Drafters
 * and tree verify, §Sampling]: at each node of the walk the target draws its
 * own token y from p = softmax(logits_row / temperature); if a child of the
 * node carries y the walk moves there, otherwise y is the round's last token
 * (at a leaf the draw is the last token).  Same law as tv_accept_residual.
 * Every row draws once, with its own uniform, by the inverse CDF (the smallest
 * y with sum_{j<=y} p(j) > u); the walk then follows these draws.
 *
 *   uniforms     device fp32 [total_rows], one per row
 *   row_tokens   device int32 [total_rows]: every row's draw
 *   path, accept_len  as tv_accept_greedy
 *   out_tokens   device int32 [total_rows]: the a_r accepted drafts, then the
 *                draw at the stopping node (a_r + 1 tokens)
 * Host checks: TV_E_TEMP, TV_E_ARG, TV_E_ROWS, TV_E_WORKSPACE.  Device checks:
 * TV_E_ORDER, TV_E_DUP_SIBLING, TV_E_UNIFORM.
 */
TV_API int tv_accept_single_draw(const tv_tree *trees, int n_req, const float *logits, int32_t vocab,
                                 float temperature, const float *uniforms, int32_t *row_tokens,
                                 int32_t *path, int32_t *accept_len, int32_t *out_tokens,
                                 int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Seeded sampled verify [Exactness, §Sampling, third paragraph; Drafters and
 * tree verify, §Sampling]: the token at sequence index t is
 * argmax_y (logits_row[y] / temperature + G_t(y)), G_t(y) = -log(-log U) with
 * U = (w + 0.5) / 2^32, w the first word of Philox4x32-10 (Salmon et al., SC
 * 2011) at counter (y, t, 0, 0) under key (seed low 32 bits, seed high 32 bits).
 * Row i (node i at position positions[r] + depth(i)) scores the token at
 * t = positions[r] + depth(i) + 1, so a request's text depends on its seed
 * and its logits only, never on what was drafted.  The walk follows these
 * draws as tv_accept_single_draw does.
 *
 *   seeds        host uint64 [n_req]
 *   positions    host int32 [n_req]: sequence index of each root's token
 *   row_tokens, path, accept_len, out_tokens  as tv_accept_single_draw
 * Host checks: TV_E_TEMP, TV_E_ARG, TV_E_ROWS, TV_E_WORKSPACE.  Device checks:
 * TV_E_ORDER, TV_E_DUP_SIBLING.
 */
TV_API int tv_accept_gumbel(const tv_tree *trees, int n_req, const float *logits, int32_t vocab,
                            float temperature, const uint64_t *seeds, const int32_t *positions,
                            int32_t *row_tokens, int32_t *path, int32_t *accept_len, int32_t *out_tokens,
                            int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Single-path rejection sampling [Algorithm and correctness contract,
 * §Single-path sampling]: the tree must be a chain (parent[i] = i - 1).  Node
 * i carries draft x_i, drawn by the caller's drafter from the proposal row
 * proposals[row_off(r) + i]; its target is p = softmax(logits of row i - 1 /
 * temperature).  Draft i is accepted iff uniforms[row_off(r) + i] < p(x_i) /
 * q(x_i) (probability min(1, p/q)).  At the first rejection one token is drawn
 * from normalize(max(p - q, 0)) by the inverse CDF with
 * uniforms[row_off(r)] and the round ends; a fully accepted chain ends with no
 * extra token.
 *
 *   proposals    device fp32 [total_rows][vocab]; the root's row is not read.
 *                Every other row must be finite, nonnegative, of unit mass
 *                (|sum - 1| <= 1e-3, summed in fp64) and nonzero at its draft
 *   uniforms     device fp32 [total_rows], all validated
 *   path, accept_len, out_tokens, out_count  as tv_accept_residual
 * Host checks: TV_E_TEMP, TV_E_ARG, TV_E_ROWS, TV_E_WORKSPACE.  Device checks:
 * TV_E_ORDER, TV_E_DUP_SIBLING, TV_E_TOKEN, TV_E_CHAIN, TV_E_UNIFORM,
 * TV_E_PROPOSAL.
 */
TV_API int tv_accept_rejection(const tv_tree *trees, int n_req, const float *logits, int32_t vocab,
                               float temperature, const float *proposals, const float *uniforms,
                               int32_t *path, int32_t *accept_len, int32_t *out_tokens, int32_t *out_count,
                               int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Optional stage timing of tv_verify_tree (for price tables and roofline
 * reports; not needed to run a round).  tv_profile_start(max_calls) creates
 * CUDA events (no device memory) and from then on each tv_verify_tree call,
 * up to max_calls of them, records TV_PROFILE_STAGES + 1 events on its stream:
 * before its first kernel and after each stage
 *   0 tree prologue + embedding/RMSNorm   1 QKV projection (tcgen05)
 *   2 QKV finalize (RoPE, K/V write)       3 tree attention (partials + merge)
 *   4 O projection (tcgen05)               5 O finalize (residual, RMSNorm)
 *   6 LM head + argmax/top-2 (tcgen05).
 * tv_profile_stop waits for the recorded events, writes per stage the SUM of
 * its durations (ms) over the recorded calls into stage_ms[0..n_stages), the
 * number of recorded calls into *n_calls, and destroys the events.  Calls
 * recorded inside a CUDA graph capture are not timed (do not profile while
 * capturing).  Process-wide, not thread-safe.
 */
#define TV_PROFILE_STAGES 7
TV_API int tv_profile_start(int max_calls);
TV_API int tv_profile_stop(float *stage_ms, int max_stages, int *n_stages, int *n_calls);

/*
 * Gated DeltaNet tree verify [Drafters and tree verify, §Tree verify through
 * recurrent layers].  The recurrent core of one Gated DeltaNet layer over a
 * draft tree: per value head the state S is a d_k x d_v fp32 matrix (keys to
 * values) and one step of the gated delta rule is
 *     S <- exp(g) (I - beta k k^T) S + beta k v^T,   o = S^T q.
 * The state after node t is the state after t's parent updated by t; the
 * state before the root is the layer's state before the round.  Value head h
 * reads key head h / (n_v_heads / n_k_heads).  The inputs are the layer's
 * per-node q, k (already normalised and scaled), v, beta in (0, 1) and
 * g <= 0 (log decay); projections and the short convolution are the caller's.
 *
 * tv_dn_verify_tree writes every node's output o_t = S_t^T q_t, and, for the
 * commit, the node's pseudo-value u_t and cumulative gate gc_t (the sum of g
 * over its root path), with which the state after any root path ending at t is
 *     exp(gc_t) S0 + sum over s on the path of exp(gc_t - gc_s) k_s u_s^T.
 *
 *   dims        host: n_k_heads >= 1, n_v_heads a multiple of it, d_k and d_v
 *               multiples of 32 up to 128 (else TV_E_UNSUPPORTED)
 *   trees       host array [n_req], as for tv_verify_tree (tokens are checked
 *               only for duplicate siblings)
 *   states      host array [n_req] of device pointers, 16-byte aligned: the
 *               layer's state of each request, fp32 [n_v_heads][d_k][d_v];
 *               read only
 *   q, k        device fp32 [total_rows][n_k_heads][d_k], 16-byte aligned
 *   v           device fp32 [total_rows][n_v_heads][d_v], 16-byte aligned
 *   beta, g     device fp32 [total_rows][n_v_heads]
 *   o, u        device fp32 [total_rows][n_v_heads][d_v]
 *   gc          device fp32 [total_rows][n_v_heads]
 * Host checks: TV_E_ARG (null or misaligned pointers), TV_E_ROWS,
 * TV_E_UNSUPPORTED.  Device checks: the tree rules.
 */
typedef struct {
    int32_t n_k_heads, n_v_heads, d_k, d_v;
} tv_dn_dims;

TV_API int tv_dn_verify_tree(const tv_dn_dims *dims, const tv_tree *trees, int n_req, float *const *states,
                             const float *q, const float *k, const float *v, const float *beta, const float *g,
                             float *o, float *u, float *gc, int32_t *dev_status, void *stream);

/*
 * Path-state commit of the Gated DeltaNet layers [Drafters and tree verify,
 * §Tree verify through recurrent layers]: for every layer and value head,
 *     S <- exp(gc_last) S + sum_{d = 0..a} exp(gc_last - gc_{p_d}) k_{p_d} u_{p_d}^T
 * over the accepted root path p_0 = 0, ..., p_a (gc_last = gc_{p_a}), i.e. the
 * state after the path's last node.  One read and one write of the state, no
 * weights.  A chain rolled back to its first m nodes is the path 0..m-1.
 *
 *   n_layers    host >= 1: layers committed in one call
 *   states      host array [n_req] of device pointers, 16-byte aligned: fp32
 *               [n_layers][n_v_heads][d_k][d_v], updated in place
 *   k           device fp32 [n_layers][total_rows][n_k_heads][d_k], 16-byte aligned
 *   u           device fp32 [n_layers][total_rows][n_v_heads][d_v], 16-byte aligned
 *   gc          device fp32 [n_layers][total_rows][n_v_heads]
 *               (u and gc as tv_dn_verify_tree wrote them, layer by layer)
 *   path, accept_len  device, from an accept walk
 * Host checks: as tv_dn_verify_tree.  Device checks: TV_E_PATH (a_r outside
 * 0..n_r - 1, path[0] != 0, or path[d] not a child of path[d - 1]); with a
 * bad path in any request no state is written.
 */
TV_API int tv_dn_commit(const tv_dn_dims *dims, const tv_tree *trees, int n_req, int n_layers, float *const *states,
                        const float *k, const float *u, const float *gc, const int32_t *path,
                        const int32_t *accept_len, int32_t *dev_status, void *stream);

/*
 * Tree verify through a stack of decoder layers [Drafters and tree verify, §The
 * round, step 2: "one forward pass of the target model runs over the whole
 * tree"; §Tree verify through recurrent layers: the model's Gated DeltaNet
 * layers].  The pages name the layer kinds, not the layers; the stack taken is
 * a pre-norm residual stack, each layer a mixer and a SwiGLU MLP:
 *
 *     x = E[token]
 *     per layer:  x = bf16( x + Mixer( bf16(RMSNorm(x) ln_mix) ) )
 *                 x = bf16( x + bf16( silu(h W_gate^T) * (h W_up^T) ) W_down^T ),
 *                     h = bf16(RMSNorm(x) ln_mlp)
 *     logits = fp32( bf16(RMSNorm(x) ln_f) W_lm^T ), argmax and top-2 gap
 *
 * Mixer of an attention layer (TV_LAYER_ATTN): the layer of tv_verify_tree
 * (QKV, RoPE at ctx + depth, tree-masked GQA attention over the layer's cache,
 * O projection); the tree rows' K/V go to its cache at slots ctx + i.
 * Mixer of a Gated DeltaNet layer (TV_LAYER_DN): [q, k, v, z, b, a] = h W_in^T
 * (rows: q, k of n_k_heads x d_k, v, z of n_v_heads x d_v, then b, a of
 * n_v_heads); per key head q and k divided by sqrt(|.|^2 + 1e-6), q also by
 * sqrt(d_k); beta = sigmoid(b), g = -softplus(a); the gated delta rule over the
 * tree as tv_dn_verify_tree (from the layer's state before the round); per
 * value head y = bf16( o / sqrt(mean(o^2) + rms_eps) dn_norm silu(z) ); the
 * mixer output is y W_out^T.
 *
 *   tv_layer     one layer, all device pointers, bf16, weights [out][in] row
 *                major (or tile-packed by tv_pack_weight when model->packed):
 *                  ln_mix, ln_mlp [hidden]
 *                  w_mix_in   attention: W_qkv [(Hq + 2 Hkv) D][hidden];
 *                             DeltaNet: W_in [2 Hk dk + 2 Hv dv + 2 Hv][hidden]
 *                  w_mix_out  attention: W_o [hidden][Hq D]; DeltaNet: W_out [hidden][Hv dv]
 *                  dn_norm    DeltaNet: [d_v]; attention: unused
 *                  w_gate_up  [2 intermediate][hidden] (gate rows, then up rows)
 *                  w_down     [hidden][intermediate]
 *   tv_stack     dims (hidden, attention heads, vocab, RoPE, eps), dn (the
 *                DeltaNet heads: d_k, d_v in {32, 64, 96, 128}), intermediate
 *                (a multiple of 64), n_layers and the host array of layers,
 *                embed / ln_f / lm_head as in tv_model, packed as in tv_model.
 *   kv           host array [n_attn_layers * n_req]: the cache of attention
 *                layer j (in layer order) for request r at kv[j * n_req + r];
 *                every layer of a request has the same ctx_len
 *   dn_states    host array [n_req] of device pointers, 16-byte aligned: fp32
 *                [n_dn_layers][n_v_heads][d_k][d_v], the states before the
 *                round (read only here; tv_commit_stack updates them)
 *   logits, argmax, top2_gap  as tv_verify_tree
 *   x_taps       device bf16 [2 n_layers + 1][total_rows][hidden], or NULL: the
 *                residual stream of every row after each residual sublayer --
 *                tap 2l is the stream entering layer l (tap 0 the embedding),
 *                tap 2l + 1 the stream after layer l's mixer, tap 2 n_layers
 *                the stream after the last layer (before the final norm).  The
 *                pages' block drafter reads such taps of the target ("the
 *                residual stream entering layers 5, 19, 33, 47 and 61")
 *                [Drafters and tree verify, §The block drafter].  Copies on
 *                the stream when given; nothing when NULL.
 *   workspace    device, >= tv_stack_workspace_size(model); also holds what
 *                tv_commit_stack needs (the DeltaNet layers' keys, pseudo-values
 *                and cumulative gates), so pass the same one to the commit
 * Host checks: TV_E_ARG, TV_E_ROWS, TV_E_CAPACITY, TV_E_WORKSPACE,
 * TV_E_UNSUPPORTED.  Device checks: the tree rules, as tv_verify_tree.
 */
#define TV_LAYER_ATTN 0
#define TV_LAYER_DN 1
typedef struct tv_layer {
    int32_t kind;
    const tv_bf16 *ln_mix;
    const tv_bf16 *w_mix_in;
    const tv_bf16 *w_mix_out;
    const tv_bf16 *dn_norm;
    const tv_bf16 *ln_mlp;
    const tv_bf16 *w_gate_up;
    const tv_bf16 *w_down;
} tv_layer;

typedef struct tv_stack {
    tv_dims dims;
    tv_dn_dims dn;
    int32_t intermediate;
    int32_t n_layers;
    const tv_layer *layers;
    const tv_bf16 *embed, *ln_f, *lm_head;
    int32_t packed;
} tv_stack;

TV_API int tv_stack_workspace_size(const tv_stack *model, size_t *bytes);
TV_API int tv_verify_stack(const tv_stack *model, const tv_kv *kv, float *const *dn_states, const tv_tree *trees,
                           int n_req, float *logits, int32_t *argmax, float *top2_gap, tv_bf16 *x_taps,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Commit of a stack verify [Drafters and tree verify, §The round, step 4: keep
 * the KV rows and the recurrent state of the accepted path]: in every
 * attention layer the KV commit of tv_commit_kv, in every Gated DeltaNet layer
 * the path-state commit of tv_dn_commit (the state after the path's last
 * node), from what tv_verify_stack left in the workspace.
 *   kv, dn_states, trees  as tv_verify_stack (the same call's)
 *   path, accept_len      device, from an accept walk on that call's argmax
 *   committed_src, new_ctx  as tv_commit_kv
 * Host checks: TV_E_ARG, TV_E_ROWS, TV_E_WORKSPACE, TV_E_UNSUPPORTED.  Device
 * checks: TV_E_PATH (nothing is written with a bad path).
 */
TV_API int tv_commit_stack(const tv_stack *model, const tv_kv *kv, float *const *dn_states, const tv_tree *trees,
                           int n_req, const int32_t *path, const int32_t *accept_len, int32_t *committed_src,
                           int32_t *new_ctx, const void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           void *stream);

/*
 * Verify prices and the StairCut cut [Drafters and tree verify, §StairCut: the
 * node count, calculated each round; §StairCut on Flash-Next, and the shared
 * price files].  Host-only: no device memory, nothing launched.
 *
 * tv_price_table holds the measured verify prices V(rows) by context class and
 * kind, and the online state that follows the live prices.  The caller owns
 * it (plain memory, no allocation); tv_price_init empties it, then the caller
 * fills n_classes, class_ctx (ascending context lengths), prior (milliseconds
 * of the measured counts, NaN elsewhere) and step_ms (ms a row past the last
 * measured count; 0: the slope of the last two counts).
 *
 * tv_price_lookup: V(rows) for a context and kind.  The context takes the
 * nearest lower class (the lowest if it is below all); rows between two
 * measured counts interpolate; rows past the last measured count extrapolate
 * as above; rows below the first take its price; a price never falls with more
 * rows (the maximum over counts 1..rows).  An observed count uses its live
 * price, the others the table's plus the learned offset of (class, kind).
 *
 * tv_price_observe: a measured verify time for (context, kind, rows): the
 * count's live price moves toward it by an exponential average of weight 0.1,
 * and the offset of (class, kind) moves by the same average of (observed -
 * table price).
 *
 * tv_staircut: the cut of one drafted candidate.  Nodes 1..n-1 are admitted in
 * the order of score (highest first, lower index on ties), each after its
 * ancestors not yet admitted; the cut sizes tried are 7, 15, 23 and 31 nodes
 * and the whole candidate, and the one maximising
 *     (1 + min(sum of min(q, 1) over kept nodes, kept)) /
 *     (V(kept + 1 rows) + draft_ms + commit_ms)
 * is kept (a chain, kind TV_KIND_CHAIN, pays (1 - q of its deepest kept node)
 * x rollback_ms instead of commit_ms; equal values keep the smaller cut).
 *   parent, q, score  host arrays [n], parent-before-child, parent[0] = -1;
 *                     q = the node's path probability
 *   keep              host int32 [n]: the kept nodes in admission order
 *                     (every prefix of it is a tree); *n_keep of them
 *   value             the maximised expected tokens per millisecond
 * Errors: TV_E_ARG (null, kind, an invalid table), TV_E_ROWS (n or rows
 * outside 1..32), TV_E_ORDER (parent order).
 */
#define TV_KIND_CHAIN 0
#define TV_KIND_TREE 1
#define TV_PRICE_MAX_CLASSES 16
#define TV_PRICE_MAX_ROWS 32
typedef struct {
    int32_t n_classes;
    int32_t class_ctx[TV_PRICE_MAX_CLASSES];
    double step_ms;
    double prior[TV_PRICE_MAX_CLASSES][2][TV_PRICE_MAX_ROWS + 1];   /* [class][kind][rows], NaN: not measured */
    double live[TV_PRICE_MAX_CLASSES][2][TV_PRICE_MAX_ROWS + 1];    /* NaN: never observed */
    double offset[TV_PRICE_MAX_CLASSES][2];
} tv_price_table;

TV_API int tv_price_init(tv_price_table *t);
TV_API int tv_price_lookup(const tv_price_table *t, int32_t context, int32_t kind, int32_t rows, double *ms);
TV_API int tv_price_observe(tv_price_table *t, int32_t context, int32_t kind, int32_t rows, double ms);
TV_API int tv_staircut(const int32_t *parent, const float *q, const float *score, int32_t n, int32_t kind,
                       const tv_price_table *t, int32_t context, double draft_ms, double commit_ms,
                       double rollback_ms, int32_t *keep, int32_t *n_keep, double *value);

/* A short English name of a status code (static storage). */
TV_API const char *tv_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* TV_H */
