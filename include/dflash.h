/*
 * dflash.h -- C ABI of the DFlash speculate-and-verify step on one GB300
 * (sm_103a), plus its DDTree draft-tree variant.
 *
 * The step follows the four stages described in the "DFlash speculative
 * decoding" glossary entry (globaladvisors.biz), section "DFlash:
 * architecture and workflow":
 *   1. the anchor is the token at the decoding frontier;
 *   2. the block-diffusion drafter fills B-1 masked positions in ONE forward
 *      pass, conditioned on target hidden states injected into the K/V of
 *      every draft layer ("DFlash, Diffusion LLMs, dLLM, MTP and Speculative
 *      Decoding: A Deep Research Report", section "Key points");
 *   3. the target verifies the whole block in one forward pass, comparing
 *      each draft token with its own argmax;
 *   4. the longest matching prefix is emitted, followed by the target's own
 *      token at the first mismatch, and the cycle restarts at the new
 *      frontier.
 * DDTree ("LLMs hit ludicrous speed ..." (joindrip.ai), DDTree paragraph)
 * replaces the single draft by a best-first tree of continuations built from
 * the drafter's per-position distributions, verified in one target pass with
 * an ancestor-only attention mask.
 *
 * Conventions shared by every call:
 *  - Pointers named *_dev are device pointers; the library never frees them.
 *    Weights are BORROWED: they must stay valid until dflash_destroy.
 *    KV caches, the hidden-state capture buffer and all scratch belong to the
 *    context and are allocated once, in dflash_create.
 *  - A context belongs to the device that was current at dflash_create; its
 *    calls must be made with that device current (else DFLASH_E_STATE and
 *    nothing is launched).
 *  - Every call only enqueues work on `stream` and returns without waiting
 *    for the GPU.  A context keeps scratch between calls, so all calls on one
 *    context must be issued on one stream (or otherwise ordered); one
 *    context per host thread.
 *  - Host-side argument checks run before any launch; on failure the call
 *    returns an error status and launches nothing.  Violations found on the
 *    device (a sequence that would overflow its cache, a tree deeper than the
 *    block) set a sticky status word instead of trapping; dflash_check reads
 *    it.  No kernel of this library traps or waits without a bound.
 *  - Token ids are int32.  Sequences are addressed by slot id in
 *    [0, max_batch); each slot keeps its committed length on the device.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (a CUDA runtime stream handle); 0 = legacy stream. */
typedef struct CUstream_st *dflash_stream_t;

typedef enum {
  DFLASH_OK = 0,
  DFLASH_E_INVALID_ARG = 1,   /* bad pointer, size, id or name */
  DFLASH_E_CAPACITY = 2,      /* request exceeds a capacity fixed at create */
  DFLASH_E_OOM = 3,           /* device allocation failed in dflash_create */
  DFLASH_E_CUDA = 4,          /* a CUDA runtime/driver call failed */
  DFLASH_E_DEVICE_CHECK = 5,  /* a device-side check failed (sticky) */
  DFLASH_E_TIMEOUT = 6,       /* a bounded device wait gave up (sticky) */
  DFLASH_E_UNSUPPORTED = 7,   /* shape/dtype combination not built */
  DFLASH_E_STATE = 8          /* call order violated (e.g. weights missing) */
} dflash_status;

enum { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_I32 = 2 };

typedef struct {
  /* target (and drafter: same width, heads, FFN, vocabulary) */
  int32_t d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  int32_t n_target_layers;
  int32_t n_draft_layers;
  int32_t n_inject;            /* number of target layers whose output is injected */
  int32_t inject_layers[16];   /* ascending 0-based target layer ids */
  float rope_theta, rms_eps;
  int32_t block_size;          /* B, 1..16 */
  /* capacities */
  int32_t max_batch;           /* sequence slots */
  int32_t max_ctx;             /* cache slots per sequence (prompt + generated + B or tree) */
  int32_t max_rows;            /* rows of one target pass (batch*q), >= max_batch*block */
  int32_t max_tree_nodes;      /* 0 or >= 2 (root + drafted nodes), <= 128 */
  int32_t dtype;               /* storage type of weights, caches, capture: DFLASH_F32 | DFLASH_BF16 */
  int32_t kv_pages;            /* paged KV cache: pages of DFLASH_PAGE_SLOTS slots in each
                                  layer's pool, shared by all slots (dflash_kv_reserve);
                                  0: every slot owns max_ctx slots of its own */
} dflash_config;

/* Cache slots per KV page (one attention key tile). */
#define DFLASH_PAGE_SLOTS 128

typedef struct dflash_ctx dflash_ctx;

/* Draft tree of one batch, all arrays device memory owned by the caller.
 * Node 0 is the root (the anchor); nodes are numbered in heap pop order, so
 * a parent always has a smaller id than its children. */
typedef struct {
  int32_t *tok;        /* [batch][max_nodes]  token id, -1 past n_nodes */
  int32_t *parent;     /* [batch][max_nodes]  parent id, -1 for the root */
  int32_t *depth;      /* [batch][max_nodes]  0 for the root, 1..B-1 */
  uint64_t *anc;       /* [batch][max_nodes][anc_words] bit m set = node m is an ancestor or self */
  int32_t *n_nodes;    /* [batch] */
  int32_t max_nodes;   /* row stride of the arrays above */
  int32_t anc_words;   /* ceil(max_nodes / 64) */
} dtree_buffers;

/* Accept modes of dflash_accept_commit. */
enum {
  DFLASH_ACCEPT_GREEDY = 0,  /* longest matching prefix + bonus (block) or tree walk */
  DFLASH_ACCEPT_ALL = 1,     /* commit every row of the pass (prompt prefill) */
  DFLASH_ACCEPT_GIVEN = 2    /* accept length and emitted token decided by the caller
                                (temperature-1 acceptance, dflash_spec_accept_sampled) */
};

/* Flags of dflash_verify. */
enum {
  DFLASH_VERIFY_LAST_ONLY = 1  /* run the lm_head on each sequence's last row only */
};

/* Creates a context: validates the configuration, allocates KV caches of
 * the target (n_target_layers) and of the drafter (n_draft_layers), the
 * capture buffer of injected hidden states and all scratch, and uploads the
 * RoPE tables.  Uses the current CUDA device.  On success *out owns them. */
DFLASH_API dflash_status dflash_create(const dflash_config *cfg, dflash_ctx **out);

/* Registers a borrowed weight tensor (row-major, device memory, dtype must be
 * the context's storage type).  Names and shapes, with d = d_model,
 * q = n_heads*head_dim, kv = n_kv_heads*head_dim, F = ffn_dim:
 *   tok_emb [vocab][d]  lm_head [vocab][d]  final_norm [d]
 *   layers.<l>.{attn_norm [d], wq [q][d], wk [kv][d], wv [kv][d], wo [d][q],
 *               ffn_norm [d], w_gate [F][d], w_up [F][d], w_down [d][F]}
 *   draft.fuse [d][n_inject*d]  draft.mask_emb [d]  draft.final_norm [d]
 *   draft.layers.<l>.{same names as a target layer}
 * The drafter shares tok_emb and lm_head with the target. */
DFLASH_API dflash_status dflash_set_weight(dflash_ctx *ctx, const char *name, const void *dev_ptr,
                                int32_t dtype, const int64_t *shape, int32_t ndim);

/* Marks sequence slot `seq_id` empty (committed length 0).  Its KV pages stay
 * mapped (dflash_kv_release returns them). */
DFLASH_API dflash_status dflash_reset_seq(dflash_ctx *ctx, int32_t seq_id, dflash_stream_t stream);

/* ---- paged KV cache --------------------------------------------------------
 * The serving-side cache behind concurrency measurements like the SGLang line
 * of "DFlash, Diffusion LLMs, dLLM, MTP and Speculative Decoding: A Deep
 * Research Report", section "DFlash benchmark results"; the report gives no
 * layout, so this one is the library's own.
 * Every target and draft layer keeps its K and V in a pool of pages
 * [page][n_kv_heads][DFLASH_PAGE_SLOTS][head_dim]; cache slot s of sequence
 * slot q lives in page table[q][s / DFLASH_PAGE_SLOTS] at row
 * s % DFLASH_PAGE_SLOTS.  One page table serves all layers and both models
 * (a slot holds the same position in each).
 * With kv_pages = 0 at create, the pool has max_batch * ceil(max_ctx / 128)
 * pages and slot q owns pages q * ceil(max_ctx / 128) + i for good.
 * With kv_pages > 0, the pool has kv_pages pages, no slot owns any, and a
 * pass over a sequence whose slots 0 .. length + rows - 1 are not all mapped
 * sets the sticky device status DFLASH_E_CAPACITY and skips that sequence.
 *
 * dflash_kv_reserve maps pages so that slot seq_id covers slots
 * 0 .. n_slots - 1, taking free pages lowest id first, and writes the new
 * table entries on `stream` (host-to-device copy; not for use inside a
 * stream capture).  Returns DFLASH_E_CAPACITY, and maps nothing, when
 * n_slots > max_ctx or the free pages do not suffice.  With kv_pages = 0 it
 * only checks n_slots <= max_ctx.
 * dflash_kv_release returns every page of seq_id to the free list and
 * unmaps it (on `stream`); with kv_pages = 0 it does nothing.  The caller
 * orders it after the last pass over that sequence.
 * dflash_kv_free_pages: pages in the free list (-1 on a null context). */
DFLASH_API dflash_status dflash_kv_reserve(dflash_ctx *ctx, int32_t seq_id, int32_t n_slots,
                                           dflash_stream_t stream);
DFLASH_API dflash_status dflash_kv_release(dflash_ctx *ctx, int32_t seq_id, dflash_stream_t stream);
DFLASH_API int32_t dflash_kv_free_pages(const dflash_ctx *ctx);

/* The page allocator behind dflash_kv_reserve on its own (host memory only,
 * no GPU): n_pages pages, max_seqs sequence slots of at most max_pages pages.
 * dflash_kv_pool_reserve grows seq's list to need ceil(n_slots / 128) pages,
 * lowest free ids first; *first_new / *n_new receive the table index of the
 * first page added and the count (0 when nothing was needed).  It returns
 * DFLASH_E_CAPACITY and changes nothing when the pages do not suffice or
 * exceed max_pages; DFLASH_E_INVALID_ARG for a bad slot or a negative count.
 * dflash_kv_pool_release frees seq's pages and returns how many it held.
 * dflash_kv_pool_pages copies seq's page ids into out[0..max_out) and returns
 * their count.  dflash_kv_pool_free: pages in the free list. */
typedef struct dflash_kv_pool dflash_kv_pool;
DFLASH_API dflash_kv_pool *dflash_kv_pool_create(int32_t n_pages, int32_t max_seqs,
                                                 int32_t max_pages);
DFLASH_API void dflash_kv_pool_destroy(dflash_kv_pool *pool);
DFLASH_API dflash_status dflash_kv_pool_reserve(dflash_kv_pool *pool, int32_t seq, int32_t n_slots,
                                                int32_t *first_new, int32_t *n_new);
DFLASH_API int32_t dflash_kv_pool_release(dflash_kv_pool *pool, int32_t seq);
DFLASH_API int32_t dflash_kv_pool_pages(const dflash_kv_pool *pool, int32_t seq, int32_t *out,
                                        int32_t max_out);
DFLASH_API int32_t dflash_kv_pool_free(const dflash_kv_pool *pool);

/* Target pass ("verify", also used for prompt prefill and plain AR steps).
 * For every b < batch, rows j < q_len[b] hold tokens[b][j] at position
 * P_b + j, where P_b is the committed length of slot seq_ids[b].  The K/V of
 * row j are written TENTATIVELY to cache slot P_b + j of every target layer
 * (the committed length does not change); attention is causal over the
 * cache and inside the block.  The residual stream after each injected
 * layer is kept in the context's capture buffer for dflash_inject_kv.
 *   tokens_dev  [batch][q] int32
 *   q_lens_dev  [batch] int32 or NULL (= q for all)
 *   argmax_dev  [batch][q] int32: target argmax of each row (ties: lowest id);
 *               -1 for rows past q_len (and, with LAST_ONLY, all but the last)
 *   margin_dev  [batch][q] float or NULL: top-1 minus top-2 logit
 *   logits_dev  [batch][q][vocab] float or NULL: debug copy of the logits
 * Requires batch*q <= max_rows and P_b + q <= max_ctx (device-checked). */
DFLASH_API dflash_status dflash_verify(dflash_ctx *ctx, int32_t batch, const int32_t *seq_ids_dev,
                            const int32_t *tokens_dev, int32_t q, const int32_t *q_lens_dev,
                            int32_t flags, int32_t *argmax_dev, float *margin_dev,
                            float *logits_dev, dflash_stream_t stream);

/* Block size B of the draft passes that follow (and of the draft slots
 * dtree_build reads), 1 <= block <= config.block_size.  The pages train the
 * drafter with a large block that carries over to smaller inference blocks
 * (Deep Research Report, "Key points": training innovations) and name
 * adaptive block sizes as a direction (its "Discussion and open problems");
 * this call lets a caller pick B per step.  dflash_verify takes its q
 * explicitly (pass q = B).  Host state only: it applies to calls made after
 * it, enqueues nothing, and a CUDA graph captured with one B replays that B.
 * The context starts at config.block_size.  DFLASH_E_INVALID_ARG outside
 * 1..config.block_size. */
DFLASH_API dflash_status dflash_set_block_size(dflash_ctx *ctx, int32_t block);

/* One block-diffusion draft pass (stage 2).  Slot j of the block of slot
 * seq_ids[b] sits at position P_b + j; slot 0 embeds anchor_dev[b], slots
 * 1..B-1 the mask embedding (B: the block size set by dflash_set_block_size,
 * initially config.block_size).  Every block position attends to the injected
 * draft context 0..P_b-1 and to all B block positions (no mask).
 *   block_dev   [batch][B] int32 out: [anchor, d_1 .. d_{B-1}] where d_j is
 *               the argmax of the shared lm_head at slot j (ties: lowest id)
 *   topk        0, or k in 1..16: also return the top-k of every slot
 *   topk_ids_dev  [batch][B-1][topk] int32 (logit descending, ties lowest id)
 *   topk_logp_dev [batch][B-1][topk] float: log-softmax values (temperature 1)
 *   logits_dev  [batch][B-1][vocab] float or NULL: debug copy */
DFLASH_API dflash_status dflash_draft_block(dflash_ctx *ctx, int32_t batch, const int32_t *seq_ids_dev,
                                 const int32_t *anchor_dev, int32_t *block_dev, int32_t topk,
                                 int32_t *topk_ids_dev, float *topk_logp_dev, float *logits_dev,
                                 dflash_stream_t stream);

/* Acceptance and commit (stage 4) of the LAST target pass on this context
 * (dflash_verify or dtree_verify, same batch and seq_ids).
 * GREEDY, linear block (tree == NULL): with d_i = block[b][i] and
 *   y_j = argmax[b][j], a = max{ j <= q_len-1 : d_i == y_{i-1} for all i <= j };
 *   emitted[b] = d_1..d_a, y_a (then -1); next_anchor[b] = y_a;
 *   accept_len[b] = a; the committed length grows by a + 1 (rows P..P+a are
 *   kept; the rest is rolled back by length).
 * GREEDY, tree: walk from the root to the child whose token equals the
 *   current node's argmax until none matches; a = path length; the accepted
 *   nodes' K/V (every target layer) are moved to slots P+1..P+a; bonus =
 *   argmax at the last node.
 * ALL (prefill): every row j < q_len is committed; accept_len[b] = q_len;
 *   next_anchor[b] = emitted[b][0] = argmax of the last row.
 * GIVEN, linear block only: accept_len_dev[b] and next_anchor_dev[b] are
 *   READ as a (clamped to 0..q_len-1) and the token emitted after d_1..d_a
 *   (e.g. dflash_spec_accept_sampled's outputs) and left unchanged;
 *   emitted[b] = d_1..d_a, that token; argmax_dev is not read (may be the
 *   block itself); the committed length grows by a + 1 as in GREEDY.
 * In every mode the committed rows are queued for dflash_inject_kv.
 *   block_dev  [batch][q] (linear) -- the verified tokens; ignored for trees
 *   argmax_dev [batch][q] from the verify call
 *   emitted_dev [batch][q] int32, accept_len_dev / next_anchor_dev [batch] */
DFLASH_API dflash_status dflash_accept_commit(dflash_ctx *ctx, int32_t batch, const int32_t *seq_ids_dev,
                                   const int32_t *block_dev, const int32_t *argmax_dev,
                                   const dtree_buffers *tree, int32_t mode,
                                   int32_t *accept_len_dev, int32_t *next_anchor_dev,
                                   int32_t *emitted_dev, dflash_stream_t stream);

/* KV injection (Deep Research Report, "Key points"): for every queued row,
 * h_cat = concat of the captured target residual streams (layer order),
 * F = W_fuse h_cat, and for every draft layer l: K = RoPE(Wk_l F) and
 * V = Wv_l F are written to the draft cache at the row's position.
 * With hidden_dev == NULL the rows queued by the last dflash_accept_commit
 * are injected (the other pointer arguments are ignored).  Otherwise rows
 * r < n_rows use hidden_dev[r] ([n_inject][d_model], storage dtype), slot
 * row_seq_dev[r] and position row_pos_dev[r] (< 0 skips the row); n_rows
 * <= max_rows. */
DFLASH_API dflash_status dflash_inject_kv(dflash_ctx *ctx, int32_t n_rows, const int32_t *row_seq_dev,
                               const int32_t *row_pos_dev, const void *hidden_dev,
                               dflash_stream_t stream);

/* ---- drafter and verifier in separate contexts ------------------------------
 * The glossary "DFlash speculative decoding" (section "Practical meaning and
 * deployment behaviour") notes that the drafter and the verifier may run on
 * different devices to overlap their work.  One context then runs the target
 * passes and commits (the verifier side), another the draft passes and the
 * injection (the drafter side); these two calls carry a commit across.
 *
 * dflash_injection_rows: device pointers to the rows the last
 * dflash_accept_commit queued for injection -- the capture buffer
 * [max_rows][n_inject][d_model], and per row its sequence slot (< 0: not
 * committed) and position -- and the row count.  They stay valid until the
 * next pass, commit or injection on this context.  Passing them (copied to
 * the drafter's device) to dflash_inject_kv's explicit-row form injects
 * exactly what dflash_inject_kv(ctx, 0, NULL, NULL, NULL) would here.
 *
 * dflash_advance_lengths: committed length of slot seq_ids_dev[b] += counts
 * (counts_dev[b] > 0; the verifier's accept_len + 1, or a prompt chunk's
 * length), so that the drafter-side context drafts at the same positions.
 * A count that would pass max_ctx leaves that length and sets the sticky
 * status DFLASH_E_CAPACITY; a bad slot sets DFLASH_E_DEVICE_CHECK. */
DFLASH_API dflash_status dflash_injection_rows(const dflash_ctx *ctx, const void **hidden_dev,
                                               const int32_t **row_seq_dev,
                                               const int32_t **row_pos_dev, int32_t *n_rows);
DFLASH_API dflash_status dflash_advance_lengths(dflash_ctx *ctx, int32_t batch,
                                                const int32_t *seq_ids_dev, const int32_t *counts_dev,
                                                dflash_stream_t stream);

/* DDTree build: per sequence, a best-first heap over prefixes of the per-slot
 * top-k lists (score = fp32 sum of log-probs in depth order; ties: shallower
 * first, then lexicographically smaller rank vector) pops `budget` nodes;
 * popping pushes the first child and the next sibling.  Node 0 = anchor.
 *   topk_ids_dev / topk_logp_dev [batch][B-1][topk] from dflash_draft_block
 *   budget + 1 <= tree->max_nodes <= max_tree_nodes */
DFLASH_API dflash_status dtree_build(dflash_ctx *ctx, int32_t batch, const int32_t *anchor_dev,
                          const int32_t *topk_ids_dev, const float *topk_logp_dev, int32_t topk,
                          int32_t budget, const dtree_buffers *tree, dflash_stream_t stream);

/* DDTree verify: one target pass over every node; node n sits at position
 * P + depth[n] and tentative cache slot P + n, and attends to the context
 * 0..P-1 plus its ancestors and itself.
 *   node_argmax_dev [batch][max_nodes] (-1 past n_nodes); margin/logits as
 *   in dflash_verify (row stride max_nodes) or NULL. */
DFLASH_API dflash_status dtree_verify(dflash_ctx *ctx, int32_t batch, const int32_t *seq_ids_dev,
                           const dtree_buffers *tree, int32_t *node_argmax_dev, float *margin_dev,
                           float *logits_dev, dflash_stream_t stream);

/* Waits for all work on the device, then returns (and clears) the sticky
 * device status word. */
DFLASH_API dflash_status dflash_check(dflash_ctx *ctx);

/* Text of the last host-side error of this context ("" if none). */
DFLASH_API const char *dflash_last_error(const dflash_ctx *ctx);

/* Device pointer to the committed length of every sequence slot [max_batch]. */
DFLASH_API const int32_t *dflash_seq_lengths(const dflash_ctx *ctx);

/* Number of kernels this context has launched so far. */
DFLASH_API int64_t dflash_launch_count(const dflash_ctx *ctx);

/* Read-only views of internal buffers for tests and tooling.
 *   "k_cache"/"v_cache"   target layer `layer`: its page pool
 *                         [pages][n_kv_heads][DFLASH_PAGE_SLOTS][head_dim]
 *   "dk_cache"/"dv_cache" draft layer `layer`: same layout
 *   "page_table"          [max_batch][ceil(max_ctx / 128)] int32 page ids (-1: unmapped)
 *   "capture"             [max_rows][n_inject][d_model] (row = b*q + j of the last pass)
 *   "fused"               [max_rows][d_model]: the fused feature F = W_fuse h_cat of the
 *                         rows of the last dflash_inject_kv (row order of that call)
 *   "gen_count"           [max_batch] int32: tokens emitted per slot since its reset
 *                         (prefill counts its first token; a step counts a + 1)
 * Element type = the storage dtype unless stated.  *bytes receives the view's size. */
DFLASH_API dflash_status dflash_debug_view(const dflash_ctx *ctx, const char *name, int32_t layer,
                                const void **dev_ptr, int64_t *bytes);

/* Debug: while dst_dev is set (non-NULL), every target pass also writes the
 * residual stream after each target layer, fp32, to
 * dst_dev[layer][row][d_model] (row = b*q + j of the pass; rows past a
 * sequence's block are left as they were).  bytes must cover
 * n_target_layers * max_rows * d_model floats, and dst_dev must be 16-byte
 * aligned (DFLASH_E_INVALID_ARG otherwise).  NULL switches it off. */
DFLASH_API dflash_status dflash_debug_trace(dflash_ctx *ctx, float *dst_dev, int64_t bytes);

/* Debug: the same trace for draft passes: while dst_dev is set, every
 * dflash_draft_block also writes the residual stream after each draft layer,
 * fp32, to dst_dev[layer][row][d_model] (row = b*B + j of the pass).  bytes
 * must cover n_draft_layers * max_rows * d_model floats, and dst_dev must be
 * 16-byte aligned.  NULL switches it off. */
DFLASH_API dflash_status dflash_debug_trace_draft(dflash_ctx *ctx, float *dst_dev, int64_t bytes);

/* Debug: while set, every dflash_draft_block also copies, per draft layer, the
 * roped queries (q_dev) and the attention output (attn_dev) of the pass, in the
 * storage dtype, to [layer][row][n_heads*head_dim] (row = b*B + j); each buffer
 * must hold n_draft_layers * max_rows * n_heads * head_dim elements (bytes_each).
 * Either may be NULL; both NULL switch it off.  With these a test can check the
 * attention of a draft layer on the exact inputs the kernel saw. */
DFLASH_API dflash_status dflash_debug_trace_draft_attn(dflash_ctx *ctx, void *q_dev, void *attn_dev,
                                                       int64_t bytes_each);

DFLASH_API void dflash_destroy(dflash_ctx *ctx);

/* ---- op-level block attention (no context) --------------------------------
 * The attention of one block-draft layer (Deep Research Report, "Key points":
 * the drafter's B block positions see the injected context; report's MTP
 * table and "Why DFlash beats EAGLE-3" item 3: bidirectional inside the
 * block), over caller-provided bf16 tensors, head_dim 128:
 *   q_dev   [batch][block][n_heads][128]
 *   k_dev, v_dev [batch][n_kv_heads][ctx_len + block][128]: slots
 *           0..ctx_len-1 hold the context, slots ctx_len.. the block's keys
 *   out_dev [batch][block][n_heads][128]
 * Query head h reads KV head h / (n_heads / n_kv_heads); scale 1/sqrt(128).
 * causal = 0: every block position sees the whole block (block draft);
 * causal = 1: block position j sees block keys 0..j (verify).
 * workspace_dev holds split-KV partials (fp32); pass at least
 * dflash_block_attention_workspace(...) bytes, or NULL / 0 to run without
 * splitting the context (slower at small batch, same result up to rounding).
 * Every pointer must be 16-byte aligned.
 * Returns DFLASH_E_INVALID_ARG for unsupported shapes (block 1..64,
 * n_heads / n_kv_heads must divide 64) and for misaligned pointers. */
DFLASH_API dflash_status dflash_block_attention(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                                int32_t ctx_len, int32_t block, int32_t causal,
                                                const void *q_dev, const void *k_dev,
                                                const void *v_dev, void *out_dev,
                                                void *workspace_dev, int64_t workspace_bytes,
                                                dflash_stream_t stream);

/* Bytes of workspace dflash_block_attention uses for these sizes on the
 * current device (0: no split needed; -1: unsupported shape). */
DFLASH_API int64_t dflash_block_attention_workspace(int32_t batch, int32_t n_heads,
                                                    int32_t n_kv_heads, int32_t ctx_len,
                                                    int32_t block);

/* The same block attention for callers that cannot allocate device memory
 * where they run it: an engine's per-request path that may only use buffers
 * from the engine's own pool, a serving loop that bans cudaMalloc after
 * start-up (it can synchronize the device and fragment memory), or a plugin
 * execute call that is handed no allocator.  The pages have no counterpart;
 * this is a library convenience.
 * Arguments and result are those of dflash_block_attention; the split-KV
 * partials go to a fixed 16 MiB array in device global memory that belongs to
 * the library image (every GPU that loads the library holds it until the
 * process exits), so nothing is allocated by this call.
 * Sizes whose partials exceed 16 MiB (dflash_block_attention_workspace(...)
 * > 16 MiB) are rejected with DFLASH_E_CAPACITY and a message on stderr.
 * The first call on a device looks up the array's device address for that
 * device; make that first call before any stream capture.  All calls share
 * the one array and it keeps the last call's contents (nothing in it needs
 * to start at zero), so calls that overlap on the GPU -- on two streams at
 * once -- race and must be serialized by the caller. */
DFLASH_API dflash_status dflash_block_attention_noalloc(int32_t batch, int32_t n_heads,
                                                        int32_t n_kv_heads, int32_t ctx_len,
                                                        int32_t block, int32_t causal,
                                                        const void *q_dev, const void *k_dev,
                                                        const void *v_dev, void *out_dev,
                                                        dflash_stream_t stream);

/* ---- temperature-1 drafting and acceptance ------------------------------------
 * The pages run DFlash at temperature 1 ("DFlash benchmark results" report: an
 * average 4.03x); at that temperature the drafter fills the block with
 * sampled tokens, and besides an exact match with the target's argmax the
 * target may also accept a draft token under a sampling rule that the page
 * names but leaves unstated ("DFlash speculative decoding" glossary, section
 * "DFlash: architecture and workflow", stages 2 and 3).  These calls implement the standard speculative rejection rule,
 * which keeps the output distributed exactly as sampling the target:
 *   d_j ~ p_j = softmax(drafter logits of slot j);
 *   d_j passes when u_j * p_j(d_j) < q_{j-1}(d_j), q_i = softmax(target logits
 *   of block row i); at the first failure one token is drawn from
 *   max(0, q_{j-1} - p_j) normalised; if all B-1 pass, from q_{B-1}.
 * Every draw takes the smallest token id whose cumulative weight, summed in id
 * order, exceeds u times the total weight.  Uniforms are inputs (u in [0, 1)).
 * Logits are fp32 row-major; -inf entries have zero weight (a row with no
 * finite entry has no mass and draws -1).  Sums run in a
 * fixed order, so equal inputs give equal outputs; a decision within fp32
 * rounding of a tie may differ from an exact evaluation.
 * Vocabulary up to 524,288 ids.  Workspaces are caller device memory, 256-byte
 * aligned, of at least the size the matching *_workspace call returns (which
 * returns -1 for unsupported sizes); nothing in them needs to start at zero.
 * All calls only enqueue work on `stream`. */

/* One draw per row from softmax(logits[row]) with uniform u[row]:
 * logits [rows][vocab] fp32, u [rows], tokens [rows] int32 (outputs).
 * rows 1..65535.  Returns DFLASH_E_INVALID_ARG on bad sizes, null pointers or
 * a short / misaligned workspace, DFLASH_E_CUDA if a launch fails. */
DFLASH_API int64_t dflash_sample_workspace(int32_t rows, int32_t vocab);
DFLASH_API dflash_status dflash_sample_rows(int32_t rows, int32_t vocab, const float *logits_dev,
                                            const float *u_dev, int32_t *tokens_dev,
                                            void *workspace_dev, int64_t workspace_bytes,
                                            dflash_stream_t stream);

/* One acceptance step for `batch` sequences of block size `block` (1..32,
 * batch * block <= 65535):
 *   draft_logits [batch][block-1][vocab]: row j-1 = the drafter's slot j (the
 *     layout dflash_draft_block returns; unused when block == 1);
 *     target_logits [batch][block][vocab]: row i = the target's logits at
 *     block row i (predicting position P + i + 1);
 *   tokens [batch][block]: slot 0 the anchor, slot j = d_j;
 *   u_accept [batch][block] (entry j tests d_j; entry 0 unused);
 *   u_resample [batch]: the uniform of the final draw.
 * Outputs: accept_len [batch] = a (accepted draft tokens, 0..block-1) and
 * emitted [batch] = the token drawn after them (residual or bonus).  A draft
 * token outside [0, vocab) fails its test.  A residual without mass (q and p
 * equal up to rounding) draws from q instead.  Errors as dflash_sample_rows. */
DFLASH_API int64_t dflash_spec_accept_workspace(int32_t batch, int32_t block, int32_t vocab);
DFLASH_API dflash_status dflash_spec_accept_sampled(
    int32_t batch, int32_t block, int32_t vocab, const float *draft_logits_dev,
    const float *target_logits_dev, const int32_t *tokens_dev, const float *u_accept_dev,
    const float *u_resample_dev, int32_t *accept_len_dev, int32_t *emitted_dev,
    void *workspace_dev, int64_t workspace_bytes, dflash_stream_t stream);

/* ---- failure-path diagnostic --------------------------------------------------
 * Enqueues one kernel that waits, with the same bounded wait every pipelined
 * kernel of the library uses, on a barrier that nothing completes.  The wait
 * gives up after about 2 seconds and records a timeout in the context's
 * sticky status word, so the next dflash_check returns DFLASH_E_TIMEOUT
 * (and clears it); the context stays usable.  The pages have no counterpart:
 * this exists to test the library's failure handling. */
DFLASH_API dflash_status dflash_debug_wait_timeout(dflash_ctx *ctx, dflash_stream_t stream);

/* ---- per-kernel timing ------------------------------------------------------
 * enable != 0 starts recording a CUDA event pair around every kernel launch of
 * this context (clearing earlier records); 0 stops recording. */
DFLASH_API dflash_status dflash_profile(dflash_ctx *ctx, int32_t enable);

/* Sums the recorded launches of one kernel class (0 GEMM, 1 attention,
 * 2 row-wise ops, 3 vocabulary reductions, 4 accept / tree; -1 all): their
 * count, total device milliseconds, and the algorithmic bytes and flops the
 * library assigns them (GEMM: weights + activations + fp32 output; other
 * classes report 0).  Waits for the recorded events. */
DFLASH_API dflash_status dflash_profile_read(dflash_ctx *ctx, int32_t kind, int64_t *launches,
                                             double *ms, double *bytes, double *flops);

/* The recorded launches of one kernel class (-1: all) one by one, in launch
 * order: device milliseconds and flops of the first max_out go to ms[] and
 * flops[] (either may be NULL).  Returns how many launches were recorded, or
 * -1 on a null context or a failed event query.  Waits for the events. */
DFLASH_API int64_t dflash_profile_list(dflash_ctx *ctx, int32_t kind, double *ms, double *flops,
                                       int64_t max_out);

/* ---- launch plans (host arithmetic only: no GPU, no context) -----------------
 * The pages prescribe no kernel design; these report the shapes this library
 * picks, so that a caller (or a test) can see them without a GPU.
 *
 * Tensor-core GEMM of M token rows by an N x K weight (K a multiple of 64)
 * on a GPU with sm_count SMs.  kind: 0 fp32 result, 1 QKV, 2 SwiGLU
 * (N = gate rows + up rows, a multiple of 128), 3 residual add, 4 store,
 * 5 injected K/V, 6 lm_head with the vocabulary reduction in the epilogue, 7 an
 * lm_head whose reduction keeps the top 2 per row only (no log-sum-exp, no
 * logits), which reduces from tensor memory in registers and so may take the
 * persistent form.
 * max_splits caps the K split.  plan_out[8] receives:
 * token rows per tile, token-row tiles, 128-row weight tiles, pipeline stages,
 * K splits (= thread-block cluster size), threads per CTA, dynamic shared
 * memory bytes, and the CTAs of the persistent form (0 when every tile has a
 * CTA of its own; else one CTA per SM walks the tiles, with the epilogue of a
 * tile overlapping the next tile's main loop: passes of more tiles than SMs
 * with tiles wider than 64 token rows, no K split, and any epilogue but the
 * general lm_head's, kind 6).  In the persistent form the R = tiles mod CTAs
 * tiles past the last full round are split along K over all CTAs (stream-K)
 * when R <= 3/4 of the CTAs, R x K / 64 >= 8 x CTAs and the kind is not 7.
 * DFLASH_E_INVALID_ARG for sizes the GEMM does not take. */
DFLASH_API dflash_status dflash_plan_gemm(int32_t sm_count, int32_t M, int32_t N, int32_t K,
                                          int32_t kind, int32_t max_splits, int32_t *plan_out);

/* Split-KV plan of the bf16 attention (head_dim 128) for `batch` sequences of
 * q_per_seq query rows over at most max_keys keys, on sm_count SMs, with at
 * least min_splits splits (the engine asks for 2 on batched passes; the op
 * entry points for 1).  plan_out[3] receives: splits, keys per split (a
 * multiple of 64; max_keys when unsplit), CTAs of the split kernel.
 * DFLASH_E_INVALID_ARG for unsupported shapes. */
DFLASH_API dflash_status dflash_plan_attention(int32_t sm_count, int32_t batch, int32_t n_heads,
                                               int32_t n_kv_heads, int32_t q_per_seq,
                                               int64_t max_keys, int32_t min_splits,
                                               int32_t *plan_out);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
