/*
 * eagle_tree.h -- C ABI of the GB300 (sm_103a) EAGLE-2 draft-tree
 * verification step.
 *
 * One verification step, as the EAGLE-2 article (sbmmt.com, "Up to 5x
 * lossless acceleration: EAGLE-2 lets an RTX 3060 generate faster than an
 * A100") describes it, is:
 *
 *   for layer = 0 .. depth-1:  [et_lm_head: draft features -> logits]
 *                              et_tree_expand      (expansion phase)
 *     (or et_tree_build: all layers in one launch, then the rerank and mask,
 *      when the draft logits of every node are available up front)
 *     (or et_static_tree: a fixed tree shape, EAGLE-1 / Medusa style)
 *   et_tree_rerank                                  (reranking phase, flatten)
 *   et_tree_mask_posids                             (attention mask, positions)
 *     (or et_tree_rerank_mask: both in one launch)
 *   et_tree_attention  (inside each target layer)   (ancestor-masked attention)
 *   et_verify_accept                                (lossless acceptance)
 *   et_kv_commit                                    (accepted rows -> KV cache)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument that names a tensor is a DEVICE pointer unless the
 *   comment says "host".  The caller owns every buffer; the library allocates
 *   nothing, keeps no pointer after a call returns, and never synchronises.
 * - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t; 0
 *   is the legacy default stream).  They do no host<->device copies, so they
 *   can be captured in a CUDA graph.
 * - Shapes and limits are checked on the host before any launch; a bad
 *   argument returns ET_ERR_INVALID_ARG / ET_ERR_UNSUPPORTED and launches
 *   nothing.  A failed launch returns ET_ERR_CUDA (cudaGetLastError is
 *   consumed).
 * - Problems only the device can see (non-finite logits, an index outside
 *   its table) are OR-ed as ET_DEV_* bits into `dev_status` (a device int32,
 *   nullable).  Kernels never trap.
 * - Workspaces: calls that take `ws` need `ws_bytes` >= the matching
 *   *_workspace_size() and a 256-byte aligned `ws` that was zero-filled once
 *   before its first use (et_workspace_init does that).  Each call leaves
 *   the counters it uses at zero again.  One workspace must not be used by
 *   two calls that can run at the same time (e.g. on two streams).
 * - Layout names: B sequences, V vocabulary, D depth, k top-k, m frontier,
 *   n kept nodes, N = n + 1 flat rows (row 0 = the root), C candidates
 *   (et_num_candidates), Hq/Hkv query/KV heads, d head dim, W = ceil(N/64).
 */
#ifndef EAGLE_TREE_H
#define EAGLE_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* = cudaStream_t's pointee */
typedef struct CUstream_st *et_stream_t;

#define ET_ABI_VERSION 2

typedef enum {
    ET_OK = 0,
    ET_ERR_INVALID_ARG = 1,   /* null pointer, shape out of range, misalignment */
    ET_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. head dim other than 64/128) */
    ET_ERR_WORKSPACE = 3,     /* ws null, misaligned or smaller than required */
    ET_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed */
    ET_ERR_TIMEOUT = 5        /* a bounded device wait gave up (reported through dev_status) */
} et_status;

/* bits OR-ed into *dev_status by kernels */
#define ET_DEV_NONFINITE   1  /* NaN (counted as -inf) or +inf (counted as FLT_MAX) in logits */
#define ET_DEV_BAD_INDEX   2  /* a node / row / token index outside its table; the entry is skipped */
#define ET_DEV_DISCONNECTED 4 /* rerank found a kept node whose parent is not kept (cannot happen
                                 for keys produced by et_tree_expand) */
#define ET_DEV_TIMEOUT     8  /* a bounded wait inside a kernel gave up */

/* Tree shape.  Limits: 1 <= topk <= 32, 1 <= m <= 32, 1 <= depth <= 16,
 * topk <= V, 1 <= n <= C, n + 1 <= 128, C <= 4096, temperature > 0. */
typedef struct {
    int32_t B;            /* sequences in the batch */
    int32_t V;            /* vocabulary size */
    int32_t depth;        /* D: number of expansion layers */
    int32_t topk;         /* k: children per expanded node */
    int32_t m;            /* frontier width: nodes expanded per layer after the first */
    int32_t n;            /* nodes kept by the rerank */
    float temperature;    /* T of the target/draft distributions in stochastic acceptance */
} et_tree_cfg;

/*
 * Device-side tree state (struct of caller-owned device pointers).
 *
 * Candidate ids are layer-major: layer-1 ids are 0..k-1 in top-k rank order;
 * the children of layer L+1 follow all ids of layer L and are numbered
 * base + slot*k + rank, slot being the parent's frontier slot (frontier
 * slots hold ascending ids).  Hence a parent's id is always smaller than its
 * children's and id order is depth order.
 */
typedef struct {
    /* candidates, [B, C] each (row stride C) */
    int32_t *cand_tok;      /* token id */
    int32_t *cand_parent;   /* parent candidate id, -1 = the root */
    float   *cand_lp;       /* fp32 log-prob of the token in the parent's draft row */
    int64_t *cand_key;      /* path value: sum of rint(lp * 2^32) over the path, saturating at
                               -(2^52-1); ranks nodes exactly like the product of confidences */
    int32_t *frontier;      /* [B, m]: ids expanded by the next layer, ascending, -1 padded */
    /* flattened kept tree, [B, N] each (row stride N); row 0 is the root */
    const int32_t *root_tok;/* [B] input: token of each root (nullable: flat_tok[:,0] = -1) */
    int32_t *flat_node;     /* candidate id of each row, -1 for the root */
    int32_t *flat_tok;      /* token of each row */
    int32_t *flat_parent;   /* flat row of the parent (< own row), -1 for the root */
    int32_t *flat_depth;    /* depth, root = 0 */
} et_tree;

typedef enum { ET_BF16 = 0, ET_F32 = 1 } et_dtype;

typedef enum {
    ET_ACCEPT_GREEDY = 0,       /* argmax match along the tree */
    ET_ACCEPT_STOCH_POINT = 1,  /* point-mass proposals: accept child x w.p. r(x)/sum(r) */
    ET_ACCEPT_STOCH_DRAFTQ = 2  /* draft-q proposals: min(1, r(x)/q(x)), residual update */
} et_accept_mode;

/* Attention problem shape (host struct). */
typedef struct {
    int32_t B, N, Hq, Hkv, d; /* Hq % Hkv == 0, 128 % (Hq/Hkv) == 0, d in {64, 128}, N <= 128 */
    et_dtype dtype;           /* of q, k/v prefix, k/v tree and out */
    float scale;              /* score scale, usually 1/sqrt(d) */
    int32_t max_prefix;       /* host upper bound of prefix_len[b] (sizes the grid) */
    int64_t kv_rows;          /* d-element rows in each of k_prefix / v_prefix (bounds check) */
    int64_t kv_head_stride;   /* rows between heads of one sequence's prefix; 0 = prefix_len[b] */
    int32_t num_splits;       /* KV splits per (sequence, head, row tile); 0 = library heuristic */
    int32_t impl;             /* 0 = auto (tcgen05 for bf16 with d = 128, else mma.sync),
                                 1 = mma.sync tensor-core path, 2 = tcgen05 path
                                 (ET_ERR_UNSUPPORTED unless bf16 and d = 128) */
    int32_t flags;            /* ET_ATTN_* bits below, 0 = none */
} et_attn_shape;

/* et_attn_shape.flags: the caller promises that q, k/v_prefix, k/v_tree,
 * kv_row0 and prefix_len are not written by the kernel launched just before
 * this call in the same stream (only the mask may come from it, as it does
 * from et_tree_rerank_mask or et_tree_build in a verification step).  The
 * tcgen05 path then streams Q and the whole unmasked prefix (QK^T, online
 * softmax and P.V of every prefix tile) without waiting for that kernel: it
 * waits only before its first tree tile, whose ancestor mask that kernel
 * writes, and before it writes out, lse or the workspace.  A prefix that
 * streams while a latency-bound kernel runs costs the step almost nothing. */
#define ET_ATTN_INPUTS_READY 1

/* Draft LM head shape (host struct), see et_lm_head. */
typedef struct {
    int32_t M;      /* feature rows (nodes being expanded), 1..64 */
    int32_t H;      /* hidden size, a multiple of 64 */
    int32_t V;      /* vocabulary */
    int64_t ldo;    /* row stride of logits in elements, >= V */
} et_lmhead_shape;

/* Static draft tree configuration (host struct), see et_static_tree. */
typedef struct {
    int32_t B, V;   /* sequences, vocabulary (V <= 32768) */
    int32_t N;      /* flat rows including the root, <= 128 */
    int32_t topk;   /* ranks used: every rank[i] < topk <= 32 (et_static_tree) */
    float temperature; /* q = softmax(draft / temperature) (et_static_tree_sampled) */
} et_static_cfg;

/* KV commit shape (host struct), see et_kv_commit. */
typedef struct {
    int32_t B, N, Hkv, d;     /* as in et_attn_shape; d * sizeof(dtype) a multiple of 16 bytes */
    int32_t path_len;         /* D + 1 (columns of path), <= 17 */
    et_dtype dtype;           /* of k/v tree, the caches and the features */
    int64_t kv_head_stride;   /* rows between heads of one sequence's cache = its capacity (> 0) */
    int64_t kv_rows;          /* d-element rows in each of k_cache / v_cache (bounds check) */
    int32_t feat_dim;         /* F: elements per feature row (0 = no features); F * sizeof(dtype) % 16 == 0 */
} et_commit_shape;

/* ---- geometry helpers (host, no device work) ---- */

/* C = k + sum_{l=2..D} min(m, width_{l-1}) * k, or -1 if cfg breaks a limit. */
int32_t et_num_candidates(const et_tree_cfg *cfg);
/* Nodes expanded by `layer` (1 for layer 0, else min(m, width of layer)), -1 if out of range. */
int32_t et_layer_expanded(const et_tree_cfg *cfg, int32_t layer);
/* First candidate id of `layer` (>= 1), -1 if out of range. */
int32_t et_layer_base(const et_tree_cfg *cfg, int32_t layer);
/* Workspace bytes for et_tree_expand and et_verify_accept with this cfg. */
size_t et_tree_workspace_size(const et_tree_cfg *cfg);
/* Workspace bytes for et_tree_attention with this shape (0 if no split merge is needed). */
size_t et_tree_attention_workspace_size(const et_attn_shape *shape);
/* Splits the attention call will use for this shape. */
int32_t et_tree_attention_splits(const et_attn_shape *shape);
/* Zero-fill a workspace on `stream` (cudaMemsetAsync). */
et_status et_workspace_init(void *ws, size_t ws_bytes, et_stream_t stream);
const char *et_status_string(et_status s);
int32_t et_abi_version(void);

/*
 * et_tree_expand -- one layer of the expansion phase (EAGLE-2 article,
 * expansion phase; node value = product of confidences along the path).
 *
 * Expanded nodes: the root at layer 0, else tree->frontier[b, 0..m_l) written
 * by the previous layer (m_l = et_layer_expanded(cfg, layer)).  For each,
 * over its fp32 draft-logit row z (length V):
 *   lp = log-softmax(z) (fp32, NaN counted as -inf);
 *   children = the k largest logits (ties: lower token id), ids
 *     et_layer_base(cfg, layer+1) + slot*k + rank;
 *   key(child) = key(parent) + rint(lp(child) * 2^32) (key(root) = 0).
 * If layer + 1 < D, the frontier of layer + 1 is then the top-m_{l+1} new
 * nodes by (key desc, id asc), written in ascending id order.
 *
 * logits      fp32 table; row r starts at logits + r * row_stride.  Device
 *             memory, or page-locked host memory that the GPU addresses
 *             (cudaHostAlloc / cudaHostRegister): the kernels then read only
 *             the rows they expand, over the host link (NVLink-C2C on
 *             Grace-Blackwell), and the node-indexed table never has to be
 *             copied whole.  Pageable host memory returns ET_ERR_INVALID_ARG
 *             and launches nothing (cudaPointerGetAttributes decides, on the
 *             host, before the launch).
 * row_stride  elements between rows (>= V).  With 16-byte aligned `logits`
 *             and row_stride % 4 == 0 the rows are read with 128-bit loads.
 * row_of_node nullable int32 [B, C + 1]: table row of each node (index 0 =
 *             the root, 1 + id = candidate id).  Null: rows are in expansion
 *             order, row = b * m_l + slot (what a draft model writes).
 * ws          et_tree_workspace_size(cfg) bytes (see conventions).
 * Kernels: V <= 32768 takes one thread-block cluster of ceil(V / 4096)
 * blocks per row when the layer has fewer than 64 rows (B * m_l), else one
 * 1024-thread block per row (et_set_expand_kernel overrides the choice: the
 * same children and frontier, log-probs equal up to the order of the softmax
 * sum); larger V takes a chunked kernel.
 */
et_status et_tree_expand(const et_tree_cfg *cfg, int32_t layer,
                         const float *logits, int64_t row_stride, const int32_t *row_of_node,
                         et_tree *tree, int32_t *dev_status,
                         void *ws, size_t ws_bytes, et_stream_t stream);

/*
 * et_tree_expand_noalloc -- et_tree_expand without a caller workspace.
 * The pages have no counterpart: this is a deployment convenience.
 *
 * Some callers have no way to obtain device scratch memory: a plugin or
 * custom operator that the host framework forbids to allocate inside its
 * execute callback, a runtime that reserves all device memory up front and
 * hands out only the tensors it manages, or code that must not call
 * cudaMalloc while a stream is being captured.  This entry point computes
 * exactly what et_tree_expand computes (same kernel, same arguments minus
 * `ws`), taking its scratch from a 4 MiB array that the library places in
 * device memory when it is loaded; it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Limit: 256-byte aligned counters (4 * (B*m_l + B) bytes) plus
 * 4 * B * m_l * ceil(V / 2048) * (2 + 2k) bytes of partials must fit in
 * 4 MiB (e.g. B*m_l <= 2900 at V = 32000, k = 10); larger shapes return
 * ET_ERR_WORKSPACE and launch nothing.
 * Set-up: the first call in each CUDA context (normally a device's primary
 * context) looks up the array's device address (cudaGetSymbolAddress) with
 * that context's device current and keeps it for that context; make that
 * first call before capturing a stream into a CUDA graph.  A context that
 * was destroyed (cudaDeviceReset) must not be followed by a new one that the
 * driver gives the same handle while this library stays loaded: the kept
 * address would then be stale.
 * Sharing: every call on a device uses the same array and leaves its
 * contents behind; each call clears the counters it needs on `stream`
 * (cudaMemsetAsync) before its kernel.  Two calls whose work can overlap
 * on the GPU (different streams, or concurrent host threads) race on the
 * array: serialise them on one stream.
 */
et_status et_tree_expand_noalloc(const et_tree_cfg *cfg, int32_t layer,
                                 const float *logits, int64_t row_stride, const int32_t *row_of_node,
                                 et_tree *tree, int32_t *dev_status, et_stream_t stream);

/*
 * et_tree_rerank -- reranking phase (EAGLE-2 article): keep the n candidates
 * with the largest (key desc, id asc) -- equal values keep the shallower
 * node, so the kept tree is connected -- and flatten them: row 0 is the
 * root, rows 1..n the kept ids ascending.  Writes tree->flat_*.
 * One CTA per sequence (histogram select over C 64-bit keys).
 */
et_status et_tree_rerank(const et_tree_cfg *cfg, et_tree *tree, int32_t *dev_status,
                         et_stream_t stream);

/*
 * et_tree_mask_posids -- attention mask and position ids of the flattened
 * tree (EAGLE-2 article, attention-mask example and position encoding).
 *
 * mask   uint64 [B, N, W]: bit j of word w of row i (LSB first) is set iff
 *        flat row 64w + j is row i or one of its ancestors; bits >= N clear.
 * posids int32 [B, N]: prefix_len[b] + flat_depth[b, i].
 * prefix_len int32 [B]: tokens already in each sequence's KV cache.
 */
et_status et_tree_mask_posids(const et_tree_cfg *cfg, const et_tree *tree,
                              const int32_t *prefix_len, uint64_t *mask, int32_t *posids,
                              et_stream_t stream);

/*
 * et_tree_rerank_mask -- et_tree_rerank followed by et_tree_mask_posids in
 * one launch (EAGLE-2 article: reranking phase, then the attention mask and
 * position encoding of the flattened tree).  Writes exactly what the two
 * calls write (tree->flat_*, mask, posids); the rerank CTA of each sequence
 * builds the mask from the parent rows it has just produced, which saves a
 * launch and a round trip through memory.  Arguments as in the two calls;
 * a parent row that does not precede its child sets ET_DEV_BAD_INDEX.
 */
et_status et_tree_rerank_mask(const et_tree_cfg *cfg, et_tree *tree, const int32_t *prefix_len,
                              uint64_t *mask, int32_t *posids, int32_t *dev_status, et_stream_t stream);

/*
 * et_tree_build -- the whole draft tree in one call: D expansion layers, then
 * the rerank with the attention mask and positions (EAGLE-2 article:
 * expansion phase layer after layer, reranking phase, attention mask and
 * position encoding).  Writes exactly what D calls of et_tree_expand (layers
 * 0..D-1) followed by et_tree_rerank_mask write, for draft logits that are
 * all available up front (a node-indexed table and row_of_node as in
 * et_tree_expand, read for the root and every frontier node).
 *
 * When V <= 32768 and the B * max_l(m_l) thread-block clusters (one per
 * sequence and frontier slot, ceil(V / 4096) blocks each) fit on the GPU at
 * once, the tree is ONE kernel launch: each cluster expands its frontier
 * slot in every layer; it waits on the device (a bounded spin on a per-layer
 * counter) until every row of the previous layer has written its children,
 * then picks the frontier itself.  One more cluster per sequence merges
 * each finished layer into the running top-n and, after the last layer,
 * writes the flat tree, mask and positions -- when n + max_l(m_l * k) <= 256;
 * otherwise the rerank follows as a second launch (et_tree_rerank_mask's
 * kernel).  When the clusters do not all fit (larger batches), it is still
 * one launch, of a work-queue form: persistent 1024-thread blocks take one
 * expanded row at a time from a counter, in layer order; a row of layer l
 * waits (bounded spin) only until its own sequence's layer-l frontier is
 * written, so different sequences' layers overlap; the last row of a
 * sequence's layer picks the next frontier, and the last row of its final
 * layer reranks the sequence and writes its mask and positions.  V > 32768
 * issues the D + 1 launches of the per-layer calls (same results).
 * et_tree_build_launches(cfg) says which.
 *
 * mask, posids, prefix_len: as in et_tree_rerank_mask; all three null skips
 *               the mask and positions (then it ends like et_tree_rerank).
 * ws            et_tree_workspace_size(cfg) bytes (see conventions); the
 *               one-launch form counts each layer's finished rows in it and
 *               leaves those counters at zero.
 * A flag wait that gives up (never expected: all clusters are resident, and
 * in the work-queue form a row waits only on rows that running blocks took
 * before it) sets ET_DEV_TIMEOUT; the tree is then invalid and so are the
 * workspace's counters (layers may have finished out of order): zero the
 * workspace again before its next use.
 */
et_status et_tree_build(const et_tree_cfg *cfg, const float *logits, int64_t row_stride,
                        const int32_t *row_of_node, et_tree *tree, const int32_t *prefix_len,
                        uint64_t *mask, int32_t *posids, int32_t *dev_status,
                        void *ws, size_t ws_bytes, et_stream_t stream);
/* Kernel launches et_tree_build makes for cfg on the current device: 1, 2 (the rerank apart) or D + 1 (V > 32768). */
int32_t et_tree_build_launches(const et_tree_cfg *cfg);

/*
 * et_set_wait_limit -- a diagnostic, not part of the method.  Sets the bound,
 * in SM clock cycles, of every device-side wait of the kernels launched
 * after the call (the mbarrier waits of et_tree_attention's tcgen05 path and
 * of et_lm_head, the frontier waits of et_tree_build); 0 or a negative value
 * restores the default of 2^32 cycles (about 2 s).  A wait that runs out
 * sets ET_DEV_TIMEOUT in dev_status; the kernel lets its copies and MMAs in
 * flight finish (with the default bound), frees its tensor memory and
 * returns, and that call's outputs are undefined.  Small values exist to
 * exercise that path.  Process-wide; returns the previous bound.
 */
int64_t et_set_wait_limit(int64_t cycles);

/*
 * et_set_expand_kernel -- a tuning and test switch, not part of the method.
 * Chooses the row code of every later expansion with V <= 32768:
 *   ET_EXPAND_AUTO (the default): et_tree_expand by the layer's row count;
 *     et_tree_build in one cluster launch when its clusters fit, else in the
 *     work-queue form;
 *   ET_EXPAND_CLUSTER: one cluster of ceil(V / 4096) blocks per row;
 *     et_tree_build in one cluster launch when its clusters fit, else as the
 *     D + 1 per-layer launches;
 *   ET_EXPAND_BLOCK: one 1024-thread block per row; et_tree_build always in
 *     the work-queue form.
 * (et_tree_expand_noalloc follows et_tree_expand.)  Every choice selects the
 * same children, frontier and kept tree; log-probs agree up to the
 * summation order of the softmax normaliser.  Process-wide; returns the
 * previous choice, or -1 (and changes nothing) for any other value.
 */
#define ET_EXPAND_AUTO    0
#define ET_EXPAND_CLUSTER 1
#define ET_EXPAND_BLOCK   2
int32_t et_set_expand_kernel(int32_t which);

/*
 * et_tree_attention -- attention of the N flattened draft rows over the KV
 * prefix plus their in-tree ancestors (EAGLE-2 article: each token sees only
 * its ancestors; EAGLE blog 1.1: one target forward verifies the draft).
 *
 *   out[b,i,h] = sum_j softmax_j(scale * q[b,i,h] . k_j) v_j,
 *   j over prefix tokens 0..prefix_len[b]-1 of KV head g = h / (Hq/Hkv) and
 *   tree rows t with mask bit (b,i,t).
 *
 * q, out        [B, N, Hq, d]  (bf16 or fp32 per shape->dtype)
 * k/v_prefix    prefix row of (b, g, j) = kv_row0[b] + g * S_b + j, S_b =
 *               shape->kv_head_stride or prefix_len[b]; rows of d elements.
 * kv_row0       int64 [B] first row of each sequence's prefix.
 * prefix_len    int32 [B], each in [0, max_prefix].
 * k/v_tree      [B, N, Hkv, d]: the tree rows' own keys/values (already
 *               rotated, like q and the prefix).
 * mask          uint64 [B, N, W] from et_tree_mask_posids.
 * lse           nullable fp32 [B, Hq, N]: natural-log log-sum-exp of the
 *               scaled scores of each row.
 * ws            et_tree_attention_workspace_size(shape) bytes, 256-byte
 *               aligned, owned by the caller, zero-filled once before its
 *               first use like every workspace (may be 0/null when that size
 *               is 0: the fp32 path or one split).  Holds the fp32 partial
 *               rows and (max, sum) pairs of the KV splits (and, on the
 *               mma.sync path, one arrival counter per row tile, which every
 *               call leaves at zero); the tcgen05 path drops the partial
 *               rows' lines from L2 once merged.  Calls that run at the same
 *               time need separate workspaces.
 * Accumulation is fp32; P is rounded to the input dtype before P.V.
 * tcgen05 path: the splits of a row tile run as one thread-block cluster,
 * at most 16 (the heuristic picks at most 8, the portable size); a bounded
 * wait that expires sets ET_DEV_TIMEOUT in dev_status and leaves that tile's
 * output undefined.
 */
et_status et_tree_attention(const et_attn_shape *shape,
                            const void *q, const void *k_prefix, const void *v_prefix,
                            const int64_t *kv_row0, const int32_t *prefix_len,
                            const void *k_tree, const void *v_tree, const uint64_t *mask,
                            void *out, float *lse, int32_t *dev_status,
                            void *ws, size_t ws_bytes, et_stream_t stream);

/*
 * et_verify_accept -- lossless acceptance walk (EAGLE blog 1.2: lossless in
 * greedy and non-greedy decoding; the non-greedy rule is the speculative
 * sampling the blog cites in 1.1).
 *
 * From row 0, children are tried in ascending flat row:
 *  GREEDY: a child is accepted iff its token is the argmax (lowest id on
 *    ties) of the current row's target logits; the bonus token is that
 *    argmax at the row where the walk stops.
 *  STOCH_POINT: p = softmax(target / T); each child is a point-mass
 *    proposal, so child x is accepted iff uniforms[b, child] < r(x) / sum(r),
 *    r = p with the tokens of the siblings rejected so far at this row
 *    removed (p(x) / (1 - R) for distinct tokens, R their mass; a repeat of a
 *    rejected token is never accepted); bonus = smallest token t whose
 *    cumulative residual mass (ascending token id) exceeds
 *    uniforms[b, 0] * sum(r).  The ratio is evaluated as
 *    e(x) / (S_rest + sum of e over x and the later distinct siblings), e the
 *    unnormalised weights and S_rest the row's weight outside every child
 *    token: sums of positive terms, so it keeps its relative precision when
 *    the rejected siblings hold almost all of the mass.
 *  STOCH_DRAFTQ: q = softmax(draft row of the current node / T); accept iff
 *    uniforms[b, child] < min(1, r(x) / q(x)), r starting at p and becoming
 *    norm(max(r - q, 0)) after each rejection (kept if that mass is 0);
 *    bonus drawn from the final r the same way.
 *
 * target_logits fp32 rows, stride target_stride; target_row_of_node
 *               nullable int32 [B, C+1] (index 1 + node, 0 = root); null:
 *               row = b * N + flat row (the target forward's output order).
 * draft_logits  (DRAFTQ only) same convention with draft_row_of_node.
 *               Both tables: device memory or page-locked host memory, as the
 *               logits of et_tree_expand (only the rows the kernels use are
 *               read).  Greedy and point-mass acceptance walk each sequence's
 *               accepted path, reading at most D + 1 target rows, when B >= 8;
 *               otherwise every flat row is read at once (fewer dependent
 *               reads at small batch).
 * uniforms      fp32 [B, N] in [0, 1) (stochastic modes; nullable for GREEDY).
 * accept_len    int32 [B]: accepted draft tokens (0..D).
 * path          int32 [B, D+1]: flat rows of the accepted path, root first, -1 padded.
 * tokens        int32 [B, D+1]: accepted draft tokens then the bonus token, -1 padded.
 * ws            et_tree_workspace_size(cfg) bytes (see conventions).
 *
 * Errors: ET_ERR_INVALID_ARG for an unknown mode, a missing tree array,
 * output, uniform table (stochastic modes) or draft table (DRAFTQ), a stride
 * below V, or target rows that are not 4-byte aligned (16-byte aligned rows
 * with a stride that is a multiple of 4 are read with 128-bit loads);
 * ET_ERR_WORKSPACE as in the conventions; ET_ERR_UNSUPPORTED when B * N
 * exceeds 65535 (one grid row per flat row).  A child whose token lies
 * outside [0, V) is never accepted (DRAFTQ also sets ET_DEV_BAD_INDEX).
 */
et_status et_verify_accept(const et_tree_cfg *cfg, et_accept_mode mode, const et_tree *tree,
                           const float *target_logits, int64_t target_stride,
                           const int32_t *target_row_of_node,
                           const float *draft_logits, int64_t draft_stride,
                           const int32_t *draft_row_of_node,
                           const float *uniforms,
                           int32_t *accept_len, int32_t *path, int32_t *tokens,
                           int32_t *dev_status, void *ws, size_t ws_bytes, et_stream_t stream);

/*
 * et_lm_head -- the draft model's logits for the nodes being expanded (EAGLE
 * blog 1.2: the draft reuses the target's LM head on the features its extra
 * decoder layer produces): logits[m, v] = sum_h features[m, h] * weight[v, h],
 * bf16 inputs, fp32 accumulation and output.  The rows feed et_tree_expand
 * as its logits table (row m = the m-th expanded node, so with row_of_node =
 * NULL the features are ordered by (sequence, frontier slot)).
 *
 * features  bf16 [M, H], row-major, 16-byte aligned.
 * weight    bf16 [V, H], row-major (the LM head), 16-byte aligned.
 * logits    fp32 [M, ldo].
 * Runs on tcgen05 tensor cores, one block per 128 vocabulary rows; bound by
 * streaming the weight once (V x H x 2 bytes).  A bounded wait that expires
 * sets ET_DEV_TIMEOUT and leaves that block's logits unwritten.  No workspace.
 */
et_status et_lm_head(const et_lmhead_shape *shape, const void *features, const void *weight, float *logits,
                     int32_t *dev_status, et_stream_t stream);

/*
 * et_static_tree -- a static draft tree (EAGLE-1 / Medusa style, which the
 * EAGLE-2 article contrasts with its dynamic tree): the shape is fixed in
 * advance as flat rows, row 0 the root and row i > 0 a child of row
 * parent[i] < i with rank rank[i]; row i's token is the rank[i]-th best
 * token (largest draft logit first, lower id on ties) of the draft logits at
 * its parent.  Writes tree->flat_tok / flat_parent / flat_depth / flat_node
 * (node = row - 1, root -1; flat_tok[:, 0] = root_tok), the same flattened
 * tree et_tree_rerank produces, so et_tree_mask_posids, et_tree_attention,
 * et_verify_accept (maps indexed by node + 1 = flat row) and et_kv_commit
 * apply unchanged.
 *
 * parent, rank  int32 [N] (device), parent[0] = -1, 0 <= rank[i] < topk.
 * logits        fp32 draft table, row_stride >= V.
 * row_of_flat   int32 [B, N]: table row of each flat row's draft logits
 *               (read only for rows that have children).
 * A malformed shape (a parent not preceding its child, a rank outside
 * [0, topk), a negative table row) sets ET_DEV_BAD_INDEX; the affected
 * tokens are -1.  One thread-block cluster of ceil(V / 4096) blocks per
 * (sequence, flat row).  No workspace.
 */
et_status et_static_tree(const et_static_cfg *cfg, const int32_t *parent, const int32_t *rank,
                         const float *logits, int64_t row_stride, const int32_t *row_of_flat,
                         et_tree *tree, int32_t *dev_status, et_stream_t stream);

/*
 * et_static_tree_sampled -- a static tree whose children are independent
 * draws from the draft distribution at their parent, q = softmax(draft /
 * temperature): row i > 0 takes the smallest token t with
 * sum_{v <= t} q(v) > uniforms[b, i] (the proposal under which the draft-q
 * acceptance rule, ET_ACCEPT_STOCH_DRAFTQ, is lossless -- the speculative
 * sampling the EAGLE blog 1.1 cites).  Shape as in et_static_tree (rank is
 * not used); writes the same flat arrays.
 *
 * uniforms  fp32 [B, N] in [0, 1); slot i draws row i (slot 0 unused).
 * ws        et_static_tree_workspace_size(cfg) bytes, 256-byte aligned, no
 *           initial contents (the per-chunk (max, sum) of every parent row).
 * Two launches: chunk statistics of the rows with children (one block per
 * 4096 tokens), then one block per child row that locates the chunk where
 * its uniform falls and rescans it.  V <= 32768.
 */
size_t et_static_tree_workspace_size(const et_static_cfg *cfg);
et_status et_static_tree_sampled(const et_static_cfg *cfg, const int32_t *parent, const float *logits,
                                 int64_t row_stride, const int32_t *row_of_flat, const float *uniforms,
                                 et_tree *tree, int32_t *dev_status, void *ws, size_t ws_bytes,
                                 et_stream_t stream);

/*
 * et_kv_commit -- after acceptance, append the accepted path to the KV cache
 * (EAGLE-2 article: the flattened tree's row 0 is the root and every row
 * attends the prefix plus its ancestors; EAGLE blog 1.1: the accepted tokens
 * of one verification forward are kept, the bonus token starts the next step).
 *
 * For each sequence b with A = accept_len[b] and rows r_i = path[b, i]
 * (r_0 = 0, the root), i = 0..A:
 *   k_cache/v_cache row kv_row0[b] + g * kv_head_stride + prefix_len[b] + i
 *       <- k_tree/v_tree[b, r_i, g, :]            for every KV head g,
 *   feat_out[b, i, :] <- features[b, r_i, :]      (rows i > A are zeroed),
 *   new_prefix_len[b] = prefix_len[b] + A + 1.
 *
 * k_tree, v_tree  [B, N, Hkv, d] (the K/V the target forward computed for the
 *                 flattened tree, already rotated).
 * accept_len, path  outputs of et_verify_accept.
 * k_cache, v_cache  rows of d elements; each sequence's heads are
 *                 kv_head_stride rows apart (its capacity); written in place.
 * kv_row0, prefix_len  as in et_tree_attention; prefix_len is read only.
 * new_prefix_len  int32 [B], must not alias prefix_len.
 * features, feat_out  [B, N, F] and [B, D+1, F] (nullable when feat_dim = 0):
 *                 the target hidden states the draft model reads next.
 * Tensors 16-byte aligned.  A path row outside [0, N), an accept_len outside
 * [0, D], or a position past the capacity sets ET_DEV_BAD_INDEX and that row
 * (or sequence) is skipped.  No workspace.
 */
et_status et_kv_commit(const et_commit_shape *shape, const void *k_tree, const void *v_tree,
                       const int32_t *accept_len, const int32_t *path, void *k_cache, void *v_cache,
                       const int64_t *kv_row0, const int32_t *prefix_len, int32_t *new_prefix_len,
                       const void *features, void *feat_out, int32_t *dev_status, et_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_TREE_H */
