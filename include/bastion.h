/*
 * bastion.h -- C ABI of the BASTION spec-tree step on one GB300 (sm_103a).
 *
 * One decode step of budget-aware tree speculative decoding with
 * block-diffusion drafting ("Bastion: Budget-Aware Speculative Decoding with
 * Tree-structured Block Diffusion Drafting", explainer page
 * gist.science/de/paper/2605.29727, section "Methodik: BASTION") runs as four
 * calls, in this order, on one CUDA stream:
 *
 *   bastion_topk_softmax  per-position marginals q_k and their top-k   (Methodik §1)
 *   bastion_tree_build    best-first prefix tree + S(N) budget stop      (Methodik §1-§3)
 *   bastion_tree_attn     tree-masked verification attention            (Problemstellung;
 *                                                                        "baumgestützte Verifizierung")
 *   bastion_accept        greedy (temperature 0) acceptance             (Experimentelle Ergebnisse)
 *
 * and, beside them:
 *
 *   bastion_tree_build_threshold  stage 2 with a confidence threshold    (FlexDraft page, "Flex-Decoding")
 *   bastion_kv_commit     the accepted path joins the context KV cache  (FlexDraft page, "Flex-Decoding")
 *   bastion_block_mask    block-diffusion drafter mask for the attention (FlexDraft page, "Attention-Tuning")
 *   bastion_fit_verify_latency, bastion_latency_table
 *                         calibration of the stage-2 cost table C(N) (Methodik §3)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array argument is a DEVICE pointer on the current device, owned and
 *   allocated by the caller.  The library never allocates, frees or copies
 *   device memory, never synchronises a stream and keeps no state besides a
 *   per-device cache of launch properties (filled by bastion_init).
 * - All work is enqueued on `stream` (NULL = the legacy default stream) and
 *   returns immediately; results are valid once the stream has reached them.
 *   The four calls may be captured into a CUDA graph once bastion_init() has
 *   run for the device outside of any capture.
 * - Host-detectable problems (NULL pointers, bad sizes, unsupported shapes,
 *   workspace too small) return an error status synchronously and enqueue
 *   nothing.  A failed launch returns BASTION_ERR_CUDA.
 * - Data-dependent problems that only the device can see (a token id >= V,
 *   n[b] outside [1, n_max], a context length beyond the cache, a page id out of
 *   range) never fault: the kernel skips the bad access, writes the documented
 *   fill value and ORs a bit into *dev_err (if dev_err is not NULL).  The
 *   caller zeroes *dev_err and reads it after its own synchronisation.
 * - Calls on different streams are independent as long as they do not share
 *   output buffers or workspaces.
 * - The accept and tree_attn workspaces must be zero-filled once when
 *   allocated; every call leaves them as it needs them, so they can be reused
 *   without clearing.  Two calls in flight at the same time must not share a
 *   workspace.
 */
#ifndef BASTION_H
#define BASTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bastion_stream_t; /* same type as cudaStream_t */

typedef enum {
  BASTION_OK = 0,
  BASTION_ERR_INVALID_ARG = 1,  /* NULL pointer, negative or inconsistent size */
  BASTION_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels handle */
  BASTION_ERR_WORKSPACE = 3,    /* workspace smaller than the *_workspace_size() */
  BASTION_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed */
  BASTION_ERR_NO_DEVICE = 5,    /* no usable sm_103 device */
  BASTION_ERR_DEVICE = 6,       /* the device error word reports bad data (bastion_error_status) */
  BASTION_ERR_TIMEOUT = 7       /* the device error word reports an expired in-kernel wait */
} bastion_status;

typedef enum { BASTION_F32 = 0, BASTION_BF16 = 1 } bastion_dtype;

/* bits of the device error word */
#define BASTION_DEVERR_TOKEN 0x1u /* a token id outside [0, V) */
#define BASTION_DEVERR_N 0x2u     /* n[b] outside [1, n_max] */
#define BASTION_DEVERR_CTX 0x4u   /* ctx_len[b] < 0 or beyond the KV cache capacity */
#define BASTION_DEVERR_PAGE 0x8u  /* a block-table page id outside [0, num_pages) */
#define BASTION_DEVERR_TIMEOUT 0x10u /* a bounded in-kernel wait expired (the call's outputs are invalid) */
#define BASTION_DEVERR_LAYOUT 0x20u  /* a kernel found its shared memory misaligned and did nothing
                                       (not expected on sm_103; the call's outputs are invalid) */

/* Limits of this build. */
#define BASTION_MAX_TOPK 32     /* k of the top-k */
#define BASTION_MAX_NODES 256   /* n_max, root included */
#define BASTION_MAX_DEPTH 32    /* K, drafter positions */
#define BASTION_MAX_VOCAB 262144

/* ABI version of this header (major * 100 + minor): 101 = 100 plus the calls
 * beside the step (threshold tree build, KV commit, drafter mask, latency
 * calibration); 102 = 101 plus the error-word helpers (bastion_read_error,
 * bastion_error_status, BASTION_ERR_DEVICE / _TIMEOUT), bastion_status_str and
 * bastion_topk_softmax_workspace_size; the four stage calls are unchanged. */
int bastion_abi_version(void);

/* Human-readable name of a status. Never NULL.  bastion_status_str is the
 * same function under a shorter name. */
const char *bastion_status_string(bastion_status s);
const char *bastion_status_str(bastion_status s);

/* Device error word helpers.  Every call takes an optional device pointer
 * dev_err to one uint32 that the kernels OR BASTION_DEVERR_* bits into; the
 * caller zeroes it (e.g. cudaMemsetAsync) and reads it after the work is done.
 *
 * bastion_read_error enqueues on `stream` an asynchronous copy of the word at
 * dev_err (device) to *host_word (host; pinned memory keeps the copy
 * asynchronous) and returns at once; *host_word is valid once the caller has
 * synchronised with the stream.  NULL pointers: BASTION_ERR_INVALID_ARG; a
 * failed copy: BASTION_ERR_CUDA.
 *
 * bastion_error_status maps a word to a status: 0 -> BASTION_OK; the
 * BASTION_DEVERR_TIMEOUT bit -> BASTION_ERR_TIMEOUT (the outputs of the call
 * that set it are invalid); any other bit -> BASTION_ERR_DEVICE (some request
 * had bad data and was skipped as documented per call). */
bastion_status bastion_read_error(const uint32_t *dev_err, uint32_t *host_word, bastion_stream_t stream);
bastion_status bastion_error_status(uint32_t word);

/* Explanation of the last error status returned on this host thread
 * (empty string if none). */
const char *bastion_last_error(void);

/* Prepare `device` (which must be an sm_103 GPU): caches its SM count and sets
 * kernel attributes.  Idempotent and thread-safe.  The stage calls run it
 * implicitly on first use of a device; call it explicitly before capturing the
 * calls into a CUDA graph. */
bastion_status bastion_init(int device);

/*
 * Stage 1 -- per-position marginals and top-k (Methodik §1: the block-diffusion
 * drafter yields per-position marginals q_k(.) in one forward pass; the tree's
 * path scores come from drafter logits, "Hauptbeiträge").
 *
 * For each of `rows` drafter rows (row r at logits + r * row_stride elements,
 * V elements, dtype f32 or bf16):
 *   q(v)   = exp(l_v - m) / sum_u exp(l_u - m)   (softmax over the whole
 *            vocabulary at temperature 1, m = max logit)
 *   lse[r] = log sum_u exp(l_u)                  (float64)
 *   ids[r, 0..k-1] the k tokens of highest logit, ordered by logit descending
 *            then token id ascending;  lg = their logits (exact, as float),
 *            q = their probabilities (float, from the float64 lse).
 * Outputs: ids int32 [rows, k], lg float [rows, k], q float [rows, k],
 * lse double [rows].  Requires 1 <= k <= min(V, 32), V <= 262144,
 * row_stride >= V.  Logits must be finite.  No workspace.  dev_err (nullable)
 * receives BASTION_DEVERR_TIMEOUT if a staged copy of the row never landed.
 */
/* Workspace bytes bastion_topk_softmax needs: always 0 (the partial results
 * of a row's CTAs meet in distributed shared memory inside one thread-block
 * cluster, so the call takes no workspace argument). */
size_t bastion_topk_softmax_workspace_size(int rows, int V, int k);

bastion_status bastion_topk_softmax(const void *logits, bastion_dtype dtype, int rows, int V,
                                    int64_t row_stride, int k, int32_t *ids, float *lg, float *q,
                                    double *lse, uint32_t *dev_err, bastion_stream_t stream);

/*
 * Stage 2 -- best-first prefix tree with the online budget stop
 * (Methodik §1 "Pfad-Bewertung": rho(i) = prod_{k=1}^{d(i)} q_k(x_ik);
 *  §2: A_hat(T) = sum_{i in T} rho(i), best-first repeatedly adds the valid node
 *  of highest rho; §3: grow until S(N) = A_hat(T_N) * L_AR / C(N) starts to fall).
 *
 * Inputs per request b (B requests, K drafter positions, k candidates each):
 *   ids/lg [B, K, k] and lse [B, K] as produced by stage 1 (row b*K + p is
 *   position p+1); root_tok [B]; ctx_len [B].
 * The root is node 0 (token root_tok[b], depth 0, rho 1) and counts in N and in
 * A_hat.  A node at depth d < K offers the k candidates of position d+1 as
 * children, rho(child) = rho(parent) * q.  Nodes are added in the order
 * rho descending, token id ascending, parent index ascending, where rho is
 * compared through log rho = (fp32 sum of the path's logits, root to leaf) -
 * (sum of the positions' lse).
 * Budget:  C == NULL: fixed, n[b] = min(n_max, nodes that exist).
 *          C != NULL: table C[0..n_max], C[n] = cost of verifying n nodes.
 *          Nodes are added unconditionally up to n_min; afterwards the next
 *          node is added only if S(n+1) >= S(n); n[b] is where it stops.
 * Outputs, rows in insertion (topological) order, unused rows i >= n[b] are
 * filled with -1 (ints), 0 (rho, mask, S_curve):
 *   n int32 [B]; parent, token, depth int32 [B, n_max]; pos int32 [B, n_max]
 *   = ctx_len[b] + depth; rho float [B, n_max]; mask uint64 [B, n_max, W],
 *   W = ceil(n_max / 64), bit j of row i set iff node j is an ancestor of i or i
 *   itself; ahat float [B] = A_hat(T_n); S float [B] = S(n) (C == NULL: C = 1);
 *   S_curve float [B, n_max] (may be NULL): S(i+1) for i < n[b].
 * Requires 1 <= n_min <= n_max <= 256, 1 <= K <= 32, 1 <= k <= 32, V <= 262144,
 * L_AR > 0.  Device errors: token id outside [0, V) (BASTION_DEVERR_TOKEN).
 */
bastion_status bastion_tree_build(const int32_t *ids, const float *lg, const double *lse, int B,
                                  int K, int k, int V, const int32_t *root_tok,
                                  const int32_t *ctx_len, int n_min, int n_max, const float *C,
                                  float L_AR, int32_t *n, int32_t *parent, int32_t *token,
                                  int32_t *depth, int32_t *pos, float *rho, uint64_t *mask,
                                  float *ahat, float *S, float *S_curve, uint32_t *dev_err,
                                  bastion_stream_t stream);

/*
 * bastion_tree_build with a confidence threshold (FlexDraft page,
 * "Flex-Decoding", selective verification: branches of low cumulative draft
 * confidence are pruned and only high-confidence prefixes are verified).
 *
 * Arguments and outputs are those of bastion_tree_build plus tau in [0, 1]:
 * past n_min, the tree also stops at the first node whose rho (the cumulative
 * draft confidence of its path, the product of its positions' q) is below
 * tau; with C != NULL whichever of the two stop rules comes first ends the
 * tree.  The test compares the node's fp32 log rho (fp32 logit sum minus the
 * float64 lse prefix, rounded to fp32) with log tau rounded to fp32.  Best-first
 * pops come in non-increasing rho, so without C the tree is the first
 * max(n_min, #{rho >= tau}) nodes of the fixed-budget tree (capped at n_max).
 * tau = 0 is bastion_tree_build.  tau outside [0, 1]: BASTION_ERR_INVALID_ARG.
 */
bastion_status bastion_tree_build_threshold(const int32_t *ids, const float *lg, const double *lse, int B, int K,
                                            int k, int V, const int32_t *root_tok, const int32_t *ctx_len, int n_min,
                                            int n_max, const float *C, float L_AR, float tau, int32_t *n,
                                            int32_t *parent, int32_t *token, int32_t *depth, int32_t *pos, float *rho,
                                            uint64_t *mask, float *ahat, float *S, float *S_curve, uint32_t *dev_err,
                                            bastion_stream_t stream);

/* Context KV cache of the verification attention. */
typedef struct {
  const void *k;              /* contiguous: [B, Hkv, L_max, d]; paged: [num_pages, Hkv, page_size, d] */
  const void *v;              /* same layout as k */
  int64_t L_max;              /* contiguous: context capacity per request; paged: ignored */
  const int32_t *block_table; /* paged: [B, max_pages] page ids (device); contiguous: NULL */
  int max_pages;              /* paged: columns of block_table */
  int num_pages;              /* paged: pages in the pool */
  int page_size;              /* paged: tokens per page: 8, 16, 32, 64 or 128 */
} bastion_kv_cache;

/* Bytes of workspace bastion_tree_attn needs for these sizes on the current
 * device (bf16).  Contiguous cache: when the context is split over several
 * CTAs, one partial (O, m, l) slot of 128 x (d + 4) floats per (request, KV
 * head, 128-row tile, split), else 0.  Paged cache: one ticket word per
 * (request, KV head, 128-row tile), then two partial slots per CTA of the
 * grid (one CTA per SM).  The value depends on the device (SM count, cluster
 * occupancy): query it on the device that runs the call.  The workspace must
 * be zero-filled once when it is allocated; every call leaves it as the next
 * one needs it (after a call that reported BASTION_DEVERR_TIMEOUT, zero it
 * again).  The f32 path uses no workspace. */
size_t bastion_tree_attn_workspace_size(int B, int n_max, int Hq, int Hkv, int d,
                                        const bastion_kv_cache *kv);

/*
 * Stage 3 -- tree-masked verification attention of the tree tokens
 * (Problemstellung: the target verifies the drafted candidates in one parallel
 * pass; "Akzeptanzlänge": tree-structured verification).
 *
 * For request b, tree node i < n[b] and query head h (KV head h / (Hq/Hkv)):
 *   out[b,i,h,:] = sum_j softmax_j(q[b,i,h,:] . key_j * scale) value_j
 * over the keys j = context positions 0..ctx_len[b]-1 of that KV head, followed
 * by the tree keys k_tree[b,j,kvh,:] of every node j whose bit is set in
 * mask[b,i,:] (its ancestors and itself).  Q/K/V are already projected and
 * position-encoded by the caller (tree positions are stage 2's pos).
 * Layouts: q, out [B, n_max, Hq, d]; k_tree, v_tree [B, n_max, Hkv, d];
 * mask [B, n_max, ceil(n_max/64)] uint64; n, ctx_len int32 [B].
 * dtype bf16: tensor-core path (tcgen05, fp32 softmax and accumulation);
 * dtype f32: exact fp32 path.  out has the input dtype; rows i >= n[b] are not
 * written.  Requires d in {64, 128}, Hq % Hkv == 0, n_max <= 256, base
 * pointers 16-byte aligned; bf16 with a paged cache: B <= 512.  ws: device
 * workspace of at least bastion_tree_attn_workspace_size() bytes, 16-byte
 * aligned, zero-filled when allocated (see there), else
 * BASTION_ERR_WORKSPACE.  bf16 work: with a contiguous cache each (request,
 * KV head, 128-row tile) streams its keys on one CTA or on a cluster of CTAs
 * that split them; with a paged cache the batch's actual work (every
 * request's KV heads x 128-row tiles x 128-key tiles) is split evenly over one
 * CTA per SM.  Device errors: BASTION_DEVERR_N, _CTX, _PAGE, _TIMEOUT.
 */
bastion_status bastion_tree_attn(const void *q, const void *k_tree, const void *v_tree,
                                 bastion_dtype dtype, int B, int n_max, int Hq, int Hkv, int d,
                                 float scale, const bastion_kv_cache *kv, const int32_t *ctx_len,
                                 const uint64_t *mask, const int32_t *n, void *out, void *ws,
                                 size_t ws_bytes, uint32_t *dev_err, bastion_stream_t stream);

/* Bytes of workspace bastion_accept needs for these sizes. */
size_t bastion_accept_workspace_size(int B, int n_max);

/*
 * Stage 4 -- greedy acceptance (Experimentelle Ergebnisse: greedy decoding,
 * temperature 0; the tree verification keeps the longest valid continuation).
 *
 * target: [B, n_max] rows of V logits (row (b,i) at target + (b*n_max+i) *
 * row_stride elements); only rows i < n[b] are read.
 *   a_i = argmax_v target[b,i,v] (lowest id on ties).  Walk from the root u = 0:
 *   while some child c of u (parent[c] == u, c < n[b]) has token[c] == a_u, go
 *   to it.  Outputs: acc_len int32 [B] accepted draft tokens (0..K);
 *   acc_nodes int32 [B, K+1] the path root first, -1 padded; acc_tok int32
 *   [B, K+1] the accepted draft tokens then the bonus token a_u of the last
 *   node, -1 padded; bonus int32 [B]; argmax_out int32 [B, n_max] (may be
 *   NULL): a_i for i < n[b], -1 beyond.
 * Requires V <= 262144 (ids fit the tie-break packing), row_stride >= V,
 * 1 <= K <= 32, n_max <= 256; target finite.  Invalid n[b]: the request's
 * outputs are -1 and BASTION_DEVERR_N is set.
 */
bastion_status bastion_accept(const void *target, bastion_dtype dtype, int B, int n_max, int V,
                              int64_t row_stride, int K, const int32_t *n, const int32_t *parent,
                              const int32_t *token, int32_t *acc_len, int32_t *acc_nodes,
                              int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                              size_t ws_bytes, uint32_t *dev_err, bastion_stream_t stream);

/*
 * bastion_accept_noalloc -- bastion_accept without a workspace argument.
 *
 * No counterpart on the pages: this is an interface convenience.  Some callers
 * cannot allocate device memory when the step runs (an engine that gives all
 * free GPU memory to its KV cache at start-up and keeps no allocator reachable
 * from the decode step, or code that must not take the implicit device
 * synchronisation cudaMalloc / cudaFree can cause).  This call needs no
 * workspace: its scratch (one ticket word per request, one 8-byte argmax slot
 * per tree node) lives in a fixed array of BASTION_ACCEPT_NOALLOC_MAX_BYTES bytes
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  It never calls cudaMalloc, cudaFree or an allocating library
 * routine.
 *
 * Arguments, layouts, results and device-error behaviour are those of
 * bastion_accept.  Sizes whose scratch (bastion_accept_workspace_size(B, n_max))
 * exceeds the array return BASTION_ERR_UNSUPPORTED with an explanation in
 * bastion_last_error().  The array's device address is looked up
 * (cudaGetSymbolAddress) once per device, with that device current, while
 * bastion_init prepares the device -- which the first call of this library on
 * a device (this one included) runs implicitly; make that first call, or
 * bastion_init, before any stream capture.  Each call clears
 * the ticket words on `stream`, then launches.  All calls share the one array:
 * calls that overlap on the GPU (different streams, or different host
 * threads, without ordering between them) race and give wrong results.
 */
#define BASTION_ACCEPT_NOALLOC_MAX_BYTES (128u * 1024u)
bastion_status bastion_accept_noalloc(const void *target, bastion_dtype dtype, int B, int n_max, int V,
                                      int64_t row_stride, int K, const int32_t *n, const int32_t *parent,
                                      const int32_t *token, int32_t *acc_len, int32_t *acc_nodes,
                                      int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out,
                                      uint32_t *dev_err, bastion_stream_t stream);

/*
 * After acceptance -- commit the accepted path's keys and values to the
 * context cache (FlexDraft page, "Flex-Decoding", decoupled execution: drafting
 * continues from the verified prefix and reuses the verification pass's KV
 * cache; BASTION page, "Das Ergebnis": each step's accepted tokens extend the
 * text).
 *
 * For request b with a = acc_len[b] and c = ctx_len[b]: for j = 0..a and every
 * KV head h, the rows k_tree[b, acc_nodes[b, j], h, :] and v_tree[...] are
 * written at context position c + j of kv (contiguous: [b, h, c + j, :];
 * paged: page block_table[b, (c + j) / page_size], slot (c + j) % page_size),
 * and ctx_out[b] = c + a + 1.  acc_nodes is bastion_accept's path, root first:
 * the root (the token the previous step emitted, keyed by this step's
 * verification pass at position c) and the a accepted draft tokens; the bonus
 * token is the next step's root.  Other cache entries are not touched.
 * Layouts: k_tree, v_tree [B, n_max, Hkv, d] (dtype elements); acc_len, ctx_len,
 * ctx_out int32 [B]; acc_nodes int32 [B, K+1]; kv as for bastion_tree_attn,
 * whose k and v buffers this call WRITES (the struct's const qualifies the
 * attention call).  ctx_out may alias ctx_len (in-place advance).
 * Requires d * sizeof(dtype) a multiple of 16 bytes, d <= 512, n_max <= 256,
 * K <= 32, B <= 65535, 16-byte aligned k_tree, v_tree, kv->k, kv->v.
 * Device errors (the request copies nothing and ctx_out[b] = ctx_len[b]):
 * acc_len[b] outside [0, K] or a path node outside [0, n_max)
 * (BASTION_DEVERR_N); ctx_len[b] < 0 or c + a beyond the cache capacity
 * (BASTION_DEVERR_CTX); a page id outside [0, num_pages) (BASTION_DEVERR_PAGE).
 */
bastion_status bastion_kv_commit(const void *k_tree, const void *v_tree, bastion_dtype dtype, int B, int n_max,
                                 int Hkv, int d, int K, const int32_t *acc_len, const int32_t *acc_nodes,
                                 const bastion_kv_cache *kv, const int32_t *ctx_len, int32_t *ctx_out,
                                 uint32_t *dev_err, bastion_stream_t stream);

/*
 * Block-diffusion drafter mask (FlexDraft page, "Attention-Tuning": mask
 * tokens appended to the clean prefix attend bidirectionally inside their
 * block and to the clean prefix, isolated from other blocks; BASTION page,
 * Methodik §1: one drafter pass fills a block of positions).
 *
 * Writes mask [B, n_max, ceil(n_max/64)] uint64 for bastion_tree_attn: for
 * request b and row i < n[b], bit j is set iff j < n[b] and
 * i / block == j / block; rows i >= n[b] are zero.  With the clean prefix as
 * the context cache and the block positions' Q/K/V as the tree tensors,
 * bastion_tree_attn then computes the drafter's attention.  n int32 [B] (device).
 * Requires 1 <= n_max <= 256, block >= 1.  Device errors: n[b] outside
 * [1, n_max] (BASTION_DEVERR_N; that request's rows are zero).
 */
bastion_status bastion_block_mask(int B, int n_max, int block, const int32_t *n, uint64_t *mask, uint32_t *dev_err,
                                  bastion_stream_t stream);

/*
 * Latency-table calibration (BASTION page, Methodik §3: the controller needs
 * C(N), the cost of a step that verifies N tree tokens, and L_AR; the pages
 * model the verification latency from memory bandwidth and compute, calibrated
 * on the device's observed runtimes).  Host functions: no GPU, no stream.
 *
 * bastion_fit_verify_latency: given m >= 3 measured verification times t[i]
 * (any unit) at tree sizes N[i] (at least two distinct), fits
 *   T_verify(N) = a + b N + c max(0, N - knee)
 * by least squares (Householder QR, float64) for every integer knee in
 * [knee_lo, knee_hi] and returns the knee with the smallest squared error --
 * the smallest knee among those within 1e-9 of the minimum, relative, or
 * 1e-12 of sum t^2 -- with abc = {a, b, c} and *sse.  Where the hinge column is
 * zero or a combination of 1 and N (to 1e-9 of its norm) the fit is the
 * straight line with c = 0.  Bad input (NULL, m < 3, knee_lo > knee_hi, a
 * non-finite t, fewer than two distinct N): BASTION_ERR_INVALID_ARG.
 *
 * bastion_latency_table: C[n] = t_draft + a + b n + c max(0, n - knee) for
 * n = 0..n_max (rounded to float: the table bastion_tree_build takes, after
 * the caller copies it to the device) and *L_AR = a + b + c max(0, 1 - knee),
 * the cost of verifying one token (a plain autoregressive step).  Requires
 * 1 <= n_max <= 256.
 */
bastion_status bastion_fit_verify_latency(const int32_t *N, const double *t, int m, int knee_lo, int knee_hi,
                                          double *abc, int32_t *knee, double *sse);
bastion_status bastion_latency_table(const double *abc, int32_t knee, double t_draft, int n_max, float *C,
                                     float *L_AR);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* BASTION_H */
