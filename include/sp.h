/*
 * libsp -- shared-prefix, prefill-only label readout on GB300 (sm_103a).
 *
 * The method (openjev-sglang article on jdon.com, sections on the request
 * flow and on what prefill-only means; LLM2Jev "shared prefix" page): one
 * shared state prefix is prefilled once, every question branch (prefix +
 * question suffix) is prefilled against the cached prefix, and each branch's
 * last position is read out as log-probabilities of a few single-token labels,
 * renormalised with a stable softmax.  There is no decode.
 *
 * This header is the whole boundary.  All entry points are plain C; every
 * pointer is either HOST memory or DEVICE memory as stated per argument; no
 * entry point allocates device memory (pools, outputs, descriptors and
 * workspaces are all owned by the caller).  Device work is enqueued on the
 * caller's stream (`stream` is a cudaStream_t; NULL = legacy default stream)
 * and is asynchronous: a returned SP_OK means the launch was accepted.
 * sp_run_pass_host also enqueues its input copies on the caller's copy
 * stream, and waits on the host for the previous pass of the input set it
 * is given; sp_check_device_error synchronises its stream.
 *
 * Errors: argument and limit errors are detected on the host BEFORE anything
 * is launched (the article's rule that every rejection happens before
 * inference).  Errors that only the device can see (an out-of-range label id,
 * a label count outside [2, 64], a bounded wait that gave up) set a sticky
 * device error word, read and cleared by sp_check_device_error().
 *
 * Threading: a plan is immutable after sp_plan_build and may be read by
 * several threads; calls that share a KV pool, output or workspace must be
 * ordered by the caller (one stream, or events).
 */
#ifndef SP_H_
#define SP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sp_status {
  SP_OK = 0,
  SP_ERR_ARG = 1,            /* bad pointer, shape, count or id (host-checked)    */
  SP_ERR_LIMIT = 2,          /* request limits: >32768 tokens per branch,
                                >262144 logical tokens per request              */
  SP_ERR_POOL_FULL = 3,      /* the plan needs more KV pages than max_pages      */
  SP_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed             */
  SP_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait gave up (device word)    */
  SP_ERR_DEVICE_BOUNDS = 6,  /* a device-side bounds check failed (device word)  */
  SP_ERR_WORKSPACE = 7       /* workspace / descriptor buffer too small          */
} sp_status;

/* Model shape of the single attention layer and the LM head.
 * n_q_heads % n_kv_heads == 0 and the group n_q_heads / n_kv_heads divides
 * 128 (grouped-query attention, contiguous groups: query head h reads KV head
 * h / group); head_dim is 64 or 128; page_size must be 16 tokens; hidden is a
 * multiple of 8 (16-byte rows); vocab >= 2. */
typedef struct sp_shape {
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t hidden;
  int32_t vocab;
} sp_shape;

/* Opaque host-side plan (token trie, segments, rounds, pages, launch lists). */
typedef struct sp_plan sp_plan;

/* Token accounting of a plan.  logical_tokens counts every branch's full
 * input, as usage is reported on both pages (cache hits do not reduce it);
 * computed_tokens counts each trie segment once plus one row per branch whose
 * final position is recomputed; reused = logical - computed. */
typedef struct sp_plan_stats {
  int64_t n_requests;
  int64_t n_branches;
  int64_t n_segments;
  int64_t n_shared_segments;
  int64_t n_rounds;
  int64_t logical_tokens;
  int64_t computed_tokens;
  int64_t reused_tokens;
  int64_t node_tokens;       /* rows of the node-token arrays q/k/v/out/lse      */
  int64_t pages_used;
  int64_t desc_bytes;        /* size of the device descriptor (sp_plan_upload)    */
  int64_t attn_workspace_bytes; /* workspace needed by the attention calls      */
  int64_t cache_hit_tokens;  /* tokens reused from the prefix cache (0 without) */
} sp_plan_stats;

/* Build a plan from the branches' full token sequences.
 *
 * Source: LLM2Jev "shared prefix" page (sharing is decided on the tokenised
 * prefix; staged submission for a cold request) and the openjev-sglang
 * article (radix cache; request limits).
 *
 *   n_branches      number of branches (candidates), >= 1
 *   req_of_branch   HOST int32[n_branches]; request id of each branch; branches
 *                   of different requests never share a segment
 *   tok_offsets     HOST int64[n_branches+1]; CSR offsets into tokens
 *   tokens          HOST int32[tok_offsets[n_branches]]; every branch >= 1 token
 *   max_pages       capacity of the caller's KV pool in pages
 *   n_sms           SM count used to size split-KV work (<= 0: 152)
 *   out             receives the plan; free with sp_plan_free
 *
 * Segments (trie nodes) are laid out in "node-token" order: requests in
 * increasing request id, each request's
 * segments in depth-first pre-order with children ordered by the smallest
 * branch index passing through them.  q/k/v/out/lse rows use that order
 * (sp_plan_segments gives each segment's first row).  Every segment starts on
 * a fresh KV page; pages are numbered 0..pages_used-1 in segment order.
 *
 * Rounds: per request, scan unscored branches in order; a branch joins the
 * round unless one of its uncached shared segments was already claimed by an
 * earlier branch of the same round; joining branches claim their uncached
 * shared segments.  Round r of the plan is the union over requests.
 *
 * Errors: SP_ERR_ARG (null pointer, bad shape, empty branch, negative request
 * id), SP_ERR_LIMIT (branch > 32768 tokens or request > 262144 logical
 * tokens), SP_ERR_POOL_FULL (pages needed > max_pages). */
sp_status sp_plan_build(const sp_shape* shape, int32_t n_branches, const int32_t* req_of_branch,
                        const int64_t* tok_offsets, const int32_t* tokens, int32_t max_pages,
                        int32_t n_sms, sp_plan** out);

void sp_plan_free(sp_plan* plan);

/* ---- prefix cache across calls ------------------------------------------
 *
 * Source: LLM2Jev "shared prefix" page, section on reusing SGLang's radix
 * cache (token prefixes whose KV exists are kept across requests, a later
 * input continues from its first uncached position, and prefixes are evicted
 * when memory is short; a hot request finds its prefix already cached), and
 * the openjev-sglang article, section on the repeated state (requests that
 * repeat a state and change only the questions read only their questions).
 *
 * A cache is a host-side radix tree of the shared segments (inner trie nodes)
 * that earlier plans computed, each owning the pool pages that hold its K/V;
 * it manages every page of the caller's pool of n_pages pages.  Rules:
 *  - a branch reuses its longest cached prefix (whole nodes and possibly the
 *    start of one more), capped one token short of its length: its last
 *    position is always computed;
 *  - the uncached remainders are planned and staged like a cold request, in
 *    groups of the branches of one request whose match ends at the same place;
 *  - the new shared segments get pool pages (the lowest run of free
 *    consecutive pages, else the lowest free pages), after evicting unpinned
 *    cache leaves least recently used first when the free pages do not
 *    suffice; leaves get no pages (no later call reads them);
 *  - sp_cache_commit inserts the new shared segments whose group's match ended
 *    on a node boundary (and whose first token is not taken by a sibling).
 * Not thread-safe: one thread uses a cache and its plans at a time.  Free
 * every plan built with a cache before the cache. */
typedef struct sp_cache sp_cache;

/* A cache over a pool of n_pages >= 1 pages (all free). */
sp_status sp_cache_create(int32_t n_pages, sp_cache** out);
void sp_cache_free(sp_cache* cache);

/* out[0..4] = cached segments, cached tokens, pages in use, free pages,
 * evictions so far. */
sp_status sp_cache_get_stats(const sp_cache* cache, int64_t out[5]);

/* sp_plan_build with a prefix cache (arguments as there; the pool is the
 * cache's).  The plan covers only the uncached remainders: node-token rows,
 * q / k / v / out / lse, exist for the new segments only; cached levels are
 * read from the pool by the attention calls.  The plan pins the cache nodes
 * it reads until sp_plan_free.  SP_ERR_POOL_FULL when eviction cannot free
 * enough pages (nothing changes then except the eviction of unpinned
 * leaves). */
sp_status sp_plan_build_cached(const sp_shape* shape, sp_cache* cache, int32_t n_branches,
                               const int32_t* req_of_branch, const int64_t* tok_offsets,
                               const int32_t* tokens, int32_t n_sms, sp_plan** out);

/* Insert the plan's new shared segments into the cache.  Call it after the
 * plan's attention calls are enqueued on the stream that later plans' calls
 * use (their kernels write the pages).  Committing twice is a no-op. */
sp_status sp_cache_commit(sp_cache* cache, sp_plan* plan);

/* ---- continuous batching across requests ---------------------------------
 *
 * Source: openjev-multimodal "performance" page, section on next steps
 * (continuous batching across requests, to raise throughput); the SGLang-JAX
 * blog translation, section on reducing scheduling overhead (the host
 * prepares the next batch while the device computes the current one) is
 * prior art for the loop around it.  The pages give no admission rule; this
 * library's reading:
 *  - a request's size is its node tokens, the positions of its token trie
 *    (every distinct prefix of its branches counted once: what its plan
 *    computes cold);
 *  - requests wait in a first-in first-out queue; a batch takes them from
 *    the head, in submission order, while its node tokens stay within
 *    max_batch_tokens and its request count within max_batch_requests; the
 *    head request always goes in, so a request larger than the budget forms
 *    a batch of its own;
 *  - request i of a batch is request id i of the batch's plan (sp_plan_build
 *    over the batch's branches), so its node rows, branches and labels
 *    follow those of requests 0 .. i-1: a caller that stores each request's
 *    inputs right after the previous one's reads a batch's inputs as one
 *    contiguous slice.
 * Requests never share K/V: a request's results do not depend on the batch it
 * runs in.  Host-only; one thread uses a batcher at a time. */
typedef struct sp_batcher sp_batcher;

/* max_batch_tokens >= 1, max_batch_requests >= 1; shape as for sp_plan_build. */
sp_status sp_batcher_create(const sp_shape* shape, int64_t max_batch_tokens,
                            int32_t max_batch_requests, sp_batcher** out);
void sp_batcher_free(sp_batcher* batcher);

/* Enqueue one request: its n_branches token sequences (HOST CSR, copied).
 * out_id (may be NULL) receives its id, 0, 1, 2, ... in submission order;
 * out_node_tokens (may be NULL) its node tokens.  SP_ERR_ARG for an empty
 * request or branch, SP_ERR_LIMIT for a branch over 32768 tokens or a
 * request over 262144 tokens (checked here, before any batch forms). */
sp_status sp_batcher_submit(sp_batcher* batcher, int32_t n_branches, const int64_t* tok_offsets,
                            const int32_t* tokens, int64_t* out_id, int64_t* out_node_tokens);

/* Requests and node tokens waiting in the queue. */
sp_status sp_batcher_pending(const sp_batcher* batcher, int32_t* n_requests,
                             int64_t* n_node_tokens);

/* Form the next batch and build its plan (max_pages, n_sms as for
 * sp_plan_build; free the plan with sp_plan_free).  On return *n_requests is
 * the batch size (0 and *out_plan NULL when the queue is empty), and, as
 * views valid until the next call: request_ids [n] (submission ids),
 * branch_off [n+1] (request i owns the plan's branches branch_off[i] ..
 * branch_off[i+1]-1) and row_off [n+1] (its node rows row_off[i] ..
 * row_off[i+1]-1).  Any view pointer may be NULL.  When the plan cannot be
 * built (SP_ERR_POOL_FULL for instance) the status is returned and the queue
 * is left unchanged. */
sp_status sp_batcher_next(sp_batcher* batcher, int32_t max_pages, int32_t n_sms,
                          sp_plan** out_plan, int32_t* n_requests, const int64_t** request_ids,
                          const int32_t** branch_off, const int64_t** row_off);

sp_status sp_plan_get_stats(const sp_plan* plan, sp_plan_stats* out);

/* Round lists: round r holds round_branches[round_offsets[r] .. round_offsets[r+1]),
 * in increasing branch order.  Views into the plan, valid until sp_plan_free. */
sp_status sp_plan_rounds(const sp_plan* plan, int32_t* n_rounds, const int32_t** round_offsets,
                         const int32_t** round_branches);

/* Segment table (views, length n_segments): request, parent (-1 for a request
 * root, or with a cache for a root under its group's cached prefix), first
 * node-token row, length, round in which it is computed, whether it is
 * shared by >= 2 branches, and the index of its first entry in the
 * descriptor's page table.  Without a cache the page table is the identity
 * (segment s owns pool pages first_page, first_page + 1, ...); with a cache
 * a shared segment's entries name the pool pages the cache gave it and a
 * leaf's entries are unused placeholders (leaves are never written to the
 * pool). */
sp_status sp_plan_segments(const sp_plan* plan, int32_t* n_segments, const int32_t** seg_req,
                           const int32_t** seg_parent, const int64_t** seg_node_start,
                           const int32_t** seg_len, const int32_t** seg_round,
                           const int32_t** seg_shared, const int32_t** seg_first_page);

/* Where each segment's rows come from (views, length n_segments): a branch
 * that passes through the segment and the position, within that branch's
 * token sequence, of the segment's first token.  Node-token row
 * seg_node_start[s] + t holds position seg_pos[s] + t of branch
 * seg_branch[s]; the caller computes q / k / v of exactly those positions.
 * With a prefix cache the positions start after the reused tokens. */
sp_status sp_plan_segment_sources(const sp_plan* plan, const int32_t** seg_branch,
                                  const int32_t** seg_pos);

/* Per-branch views (length n_branches): segment holding the last token, the
 * node-token row of the last token (the readout position), the branch's
 * round, and 1 when the last row is recomputed because it was cached before
 * the branch's round (the final scoring position is always computed). */
sp_status sp_plan_branches(const sp_plan* plan, const int32_t** branch_last_seg,
                           const int64_t** branch_last_row, const int32_t** branch_round,
                           const int32_t** branch_recompute);

/* Host view of the device descriptor image (what sp_plan_upload copies):
 * a header of byte offsets and counts followed by the segment table, page
 * table, ancestor chains, append list, tile list and merge list. */
sp_status sp_plan_descriptor(const sp_plan* plan, const void** data, size_t* bytes);

/* Launch lists of one call (kind 0 = sp_prefix_attn, 1 = sp_branch_attn,
 * 2 = sp_tree_attn) of
 * `round` (or SP_ALL_ROUNDS): info[0..6] = append offset, appends, tile offset, tiles, merge
 * offset, merges (entries of the descriptor lists), partial slots used. */
sp_status sp_plan_call_info(const sp_plan* plan, int32_t round, int32_t kind, int64_t info[7]);

/* Copy the plan's device descriptor (stats.desc_bytes bytes) into the
 * caller's DEVICE buffer dev_desc (>= 256-byte aligned) on `stream`.  The host
 * source lives in the plan: keep the plan alive until the copy completes. */
sp_status sp_plan_upload(const sp_plan* plan, void* dev_desc, size_t bytes, void* stream);

#define SP_ALL_ROUNDS (-1)

/* Shared-prefix attention for the segments first computed in `round`.
 *
 * sp_prefix_attn handles the shared segments claimed in the round (the
 * article's shared-prefix prefill, computed once); sp_branch_attn handles the
 * branches' own suffixes (the branch prefill against the cached prefix) and
 * recomputed final rows; sp_tree_attn handles both in one launch.  Each
 * computes causal softmax attention of every new row over its ancestor
 * segments and its own segment (causal), scale 1/sqrt(head_dim), the levels
 * combined with a log-sum-exp merge.  A level computed by the same call is
 * read from k / v; every other level from the pool, where the call that
 * computed it wrote it (every call writes the K/V of the shared segments it
 * computes into their pool pages; leaves are read by no later call and are
 * not written).
 *
 *   dev_desc  DEVICE, the uploaded descriptor of this plan
 *   round     0 <= round < n_rounds: the segments first computed in that
 *             round; calls must run in round order, and the prefix call of a
 *             round before its branch call.  SP_ALL_ROUNDS (-1): the work of
 *             every round in one call (the prefix call before the branch
 *             call); same results, fewer launches for a one-shot pass.
 *   q         DEVICE bf16 [node_tokens, n_q_heads, head_dim]
 *   k, v      DEVICE bf16 [node_tokens, n_kv_heads, head_dim]
 *   kv_pool   DEVICE bf16, per page: K as [n_kv_heads][page_size][head_dim],
 *             then V as [n_kv_heads][page_size][head_dim]
 *             (page p starts at element p * 2 * n_kv_heads * page_size * head_dim;
 *             the pool holds at least stats.pages_used pages)
 *   out       DEVICE bf16 [node_tokens, n_q_heads, head_dim]; rows of this
 *             call's segments are written (round to nearest even)
 *   lse       DEVICE fp32 [node_tokens, n_q_heads]; natural-log sum of exp of
 *             the scaled scores of each written row
 *   workspace DEVICE, >= stats.attn_workspace_bytes, 256-byte aligned
 * All device pointers 16-byte aligned. */
sp_status sp_prefix_attn(const sp_plan* plan, const void* dev_desc, int32_t round, const void* q,
                         const void* k, const void* v, void* kv_pool, void* out, float* lse,
                         void* workspace, size_t ws_bytes, void* stream);

sp_status sp_branch_attn(const sp_plan* plan, const void* dev_desc, int32_t round, const void* q,
                         const void* k, const void* v, void* kv_pool, void* out, float* lse,
                         void* workspace, size_t ws_bytes, void* stream);

/* sp_prefix_attn and sp_branch_attn of `round` (or SP_ALL_ROUNDS) as one
 * launch: every segment of the call is read from k / v, so the branches need
 * not wait for the prefix's pool writes.  With SP_ALL_ROUNDS the whole trie
 * (the LLM2Jev page's staged rounds included) is one launch whose tiles fill
 * the GPU without split parts.  Arguments as above. */
sp_status sp_tree_attn(const sp_plan* plan, const void* dev_desc, int32_t round, const void* q,
                       const void* k, const void* v, void* kv_pool, void* out, float* lse,
                       void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes for sp_label_logprobs with n_branches rows. */
size_t sp_label_workspace_bytes(int32_t n_branches, int32_t vocab, int32_t n_sms);

/* Final-position LM-head readout (openjev-sglang article, prefill-only
 * section: log-probabilities of the requested label ids at the last position):
 *
 *   logits[n, v] = sum_k h[n, k] W[v, k];  lse[n] = ln sum_v exp(logits[n, v])
 *   logprobs[j]  = logits[n(j), label_ids[j]] - lse[n(j)]
 *
 * computed in one streaming pass over W with tensor cores; logits are never
 * written to memory.
 *
 *   h          DEVICE bf16 [N, H] (row-major), final hidden states
 *   W          DEVICE bf16 [V, H] (row-major), LM head
 *   N          1 <= N <= 4096 branches;  H: multiple of 8;  V >= 2
 *   label_off  DEVICE int32 [N+1] CSR offsets (label_off[0] = 0)
 *   label_ids  DEVICE int32 [n_labels] with 0 <= id < V
 *   n_labels   label_off[N] (host copy of the total)
 *   logprobs   DEVICE fp32 [n_labels];  lse: DEVICE fp32 [N]
 *   workspace  DEVICE, >= sp_label_workspace_bytes(N, V, n_sms), 16-byte aligned
 * Device-side checks: an id outside [0, V) yields NaN and SP_ERR_DEVICE_BOUNDS. */
sp_status sp_label_logprobs(const void* h, const void* W, int32_t N, int32_t H, int32_t V,
                            const int32_t* label_off, const int32_t* label_ids, int32_t n_labels,
                            float* logprobs, float* lse, void* workspace, size_t ws_bytes,
                            void* stream);

/* Variant of sp_label_logprobs that allocates nothing and takes no workspace.
 *
 * For callers that cannot allocate device memory: serving loops that hand out
 * every device buffer from one arena sized at start-up and allow no
 * allocation afterwards (so memory use stays fixed and no allocation call
 * synchronises the device in the middle of a request), and plain C host
 * programs that link only this library and own no device allocator of their
 * own.  Such a caller still passes its inputs and outputs.
 *
 * No counterpart in the pages: this is a property of this library only.
 *
 * The readout's scratch (one partial max / sum-of-exp pair per CTA and
 * branch, and two counters, the grid barrier's and the one that hands out
 * the last vocabulary tiles, which each call zeroes before its launch) lives in a static device array of SP_NOALLOC_SCRATCH_BYTES inside
 * the library; every GPU that loads the library holds it until the process
 * exits.  Limit: N <= SP_NOALLOC_MAX_BRANCHES; a larger N returns
 * SP_ERR_WORKSPACE and launches nothing.  The first call on each device looks
 * up the array's device address (a runtime query, no allocation); make that
 * first call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents; the only parts that must start at zero,
 * the two counters, are cleared by each call on its stream before its launch,
 * and every other entry a call reads is written by that call.  Calls that can
 * overlap on the GPU (different streams without ordering, or several threads)
 * race on the array and must be serialised by the caller.  Arguments, results
 * and other errors are those of sp_label_logprobs. */
#define SP_NOALLOC_MAX_BRANCHES 1024
#define SP_NOALLOC_SCRATCH_BYTES (256u * 1024u * 8u + 256u)
sp_status sp_label_logprobs_noalloc(const void* h, const void* W, int32_t N, int32_t H, int32_t V,
                                    const int32_t* label_off, const int32_t* label_ids,
                                    int32_t n_labels, float* logprobs, float* lse, void* stream);

/* Stable softmax over each branch's labels (openjev-sglang article, request
 * flow step 5 and the worked yes/no example):
 *   probs[j] = exp(logprobs[j] - m) / sum_i exp(logprobs[i] - m), m = branch max
 *   argmax[n] = index (within the branch) of the largest logprob; lowest on ties.
 *   logprobs  DEVICE fp32 [label_off[N]];  label_off: DEVICE int32 [N+1]
 *   probs     DEVICE fp32 [label_off[N]];  argmax: DEVICE int32 [N]
 * Each branch needs 2..64 labels (the article's option limits); otherwise its
 * outputs are NaN / -1 and SP_ERR_DEVICE_BOUNDS is raised. */
sp_status sp_label_softmax(const float* logprobs, const int32_t* label_off, int32_t N, float* probs,
                           int32_t* argmax, void* stream);

/* Question types (openjev-sglang article, section on the three question
 * types): a yes/no ("noul") question, a choice among options, and a score
 * over ordered levels. */
#define SP_QTYPE_NOUL 0
#define SP_QTYPE_CHOICE 1
#define SP_QTYPE_SCORE 2

/* The label softmax of sp_label_softmax fused with the question-type result
 * and the confidence value, one question per branch whose options are the
 * branch's labels (openjev-sglang article: request flow step 5, the three
 * question types, and the confidence section):
 *
 *   probs, argmax     exactly as sp_label_softmax
 *   value[n]          NOUL:   probs of the branch's first label (P(yes))
 *                     CHOICE: probs of the argmax label (the chosen option's
 *                             probability; the option itself is argmax[n])
 *                     SCORE:  sum_i i * probs[i], i = 0 .. k-1
 *   confidence[n]     1 - H(p) / ln k, H the entropy in nats (0 ln 0 = 0)
 *
 *   logprobs   DEVICE fp32 [label_off[N]];  label_off: DEVICE int32 [N+1]
 *   qtype      DEVICE int32 [N], each SP_QTYPE_*
 *   probs      DEVICE fp32 [label_off[N]];  argmax: DEVICE int32 [N]
 *   value, confidence  DEVICE fp32 [N]
 * Device-side checks: a branch with a label count outside 2..64 gets NaN /
 * -1 outputs, a qtype outside the three codes a NaN value; both raise
 * SP_ERR_DEVICE_BOUNDS.  One launch, one warp per branch. */
sp_status sp_label_decide(const float* logprobs, const int32_t* label_off, const int32_t* qtype,
                          int32_t N, float* probs, int32_t* argmax, float* value,
                          float* confidence, void* stream);

/* Questions assembled from yes/no candidate branches (LLM2Jev page: each
 * choice option and each score level is its own yes/no input, and the final
 * answers are read after normalisation).  Question q owns the consecutive
 * branches cand_off[q] .. cand_off[q+1]-1; y_c is candidate branch c's
 * probability of its first label ("yes"), read from `probs` (the output of
 * sp_label_softmax or sp_label_decide).
 *
 *   CHOICE / SCORE (2..64 candidates):  dist_c = y_c / sum y over the question
 *       argmax[q] = index within the question of the largest y (lowest on ties)
 *       value[q]  = dist of the argmax (CHOICE) or sum_i i * dist_i (SCORE)
 *       confidence[q] = 1 - H(dist) / ln K
 *   NOUL (exactly 1 candidate):  dist = value = y;  argmax = 0;
 *       confidence = 1 - H(y, 1 - y) / ln 2
 *
 *   probs      DEVICE fp32 [label_off[n_branches]];  label_off: DEVICE int32 [n_branches+1]
 *   cand_off   DEVICE int32 [n_questions+1], cand_off[0] = 0,
 *              cand_off[n_questions] <= n_branches
 *   qtype      DEVICE int32 [n_questions]
 *   dist       DEVICE fp32 [cand_off[n_questions]];  argmax: DEVICE int32 [n_questions]
 *   value, confidence  DEVICE fp32 [n_questions]
 * Device-side checks: a candidate count that does not fit the type, a
 * qtype outside the three codes, or candidates past n_branches give NaN /
 * -1 outputs for that question and raise SP_ERR_DEVICE_BOUNDS.  The
 * normalisation is this library's reading: the page prints no formula. */
sp_status sp_candidate_decide(const float* probs, const int32_t* label_off, int32_t n_branches,
                              const int32_t* cand_off, const int32_t* qtype, int32_t n_questions,
                              float* dist, int32_t* argmax, float* value, float* confidence,
                              void* stream);

/* Multi-token option scoring with optional label-prior calibration
 * (openjev-multimodal "performance" page, section on next steps, which
 * names both as planned work that changes the probabilities; the pages give
 * no formula, so this is the library's reading):
 *
 *   scores[o]  = sum of row_logprobs[r], r = opt_off[o] .. opt_off[o+1]-1:
 *                the option's joint log-probability by the chain rule, its
 *                rows being the log-probability of each option token at the
 *                position before it (sp_label_logprobs with one label per
 *                row: the last prompt position for the first token, the
 *                previous option token's position for the others)
 *   probs[o]   = exp(x_o - m) / sum_i exp(x_i - m) over the options of o's
 *                question, x_o = scores[o] - prior[o] (prior NULL: 0), m the
 *                question's maximum; the prior is a per-option log-probability
 *                such as the same readout on a content-free input (the
 *                diagonal form of contextual calibration)
 *   argmax[q]  = index within question q of the largest x; lowest on ties
 *
 * A one-token option without a prior is exactly the label softmax.
 *   row_logprobs  DEVICE fp32 [n_rows]
 *   opt_off       DEVICE int32 [n_opts+1]: option o owns rows opt_off[o] .. opt_off[o+1]-1
 *   q_off         DEVICE int32 [n_questions+1]: question q owns options
 *                 q_off[q] .. q_off[q+1]-1; q_off[n_questions] <= n_opts
 *   prior         DEVICE fp32 [n_opts] or NULL
 *   scores, probs DEVICE fp32 [n_opts];  argmax: DEVICE int32 [n_questions]
 * Device-side checks: a question with an option count outside 2..64, an
 * option with no rows or with rows outside [0, n_rows), or options past
 * n_opts give NaN / -1 outputs for that question and raise
 * SP_ERR_DEVICE_BOUNDS.  One launch, one warp per question.  SP_ERR_ARG for
 * null pointers (other than prior) or n_rows < 1, n_opts < 2, n_questions < 1. */
sp_status sp_option_softmax(const float* row_logprobs, int32_t n_rows, const int32_t* opt_off,
                            int32_t n_opts, const int32_t* q_off, int32_t n_questions,
                            const float* prior, float* scores, float* probs, int32_t* argmax,
                            void* stream);

/* One whole pass of the path in one call: sp_plan_build over the branches,
 * sp_plan_upload, one sp_tree_attn call for the whole trie (SP_ALL_ROUNDS),
 * sp_label_logprobs and sp_label_softmax, all enqueued on `stream` (the
 * openjev-sglang article's request flow: shared prefix and branches prefilled,
 * label log-probabilities read at each branch's last position, renormalised).
 * For callers that drive the path from C, or want its host work in one call.
 *   HOST    req_of_branch, tok_offsets, tokens: as for sp_plan_build
 *   DEVICE  q, k, v: node_rows rows in the plan's node-token order (the order
 *           sp_plan_build documents; node_rows must equal its node tokens)
 *           kv_pool: pool_pages pages; out, lse: node_rows rows
 *           desc: desc_bytes, 256-byte aligned; attn_ws: attn_ws_bytes
 *           h [n_branches, shape->hidden], W [shape->vocab, shape->hidden],
 *           label_off [n_branches+1], label_ids [n_labels], logprobs and
 *           probs [n_labels], lse_vocab and argmax [n_branches],
 *           lm_ws: lm_ws_bytes (sp_label_workspace_bytes(n_branches, vocab, 0))
 *   stats   HOST, may be NULL: the pass's plan statistics, filled whenever
 *           the plan was built (also on SP_ERR_WORKSPACE and SP_ERR_POOL_FULL,
 *           where pages_used gives the pool size needed)
 * Every capacity is checked before the first launch: SP_ERR_POOL_FULL when
 * the plan needs more than pool_pages pages, SP_ERR_WORKSPACE when desc_bytes,
 * attn_ws_bytes or lm_ws_bytes is short (stats gives desc_bytes and
 * attn_workspace_bytes; nothing is launched then), SP_ERR_ARG when node_rows
 * differs from the plan's node tokens or when the readout's arguments fail
 * sp_label_logprobs' checks (those come first, before the plan); other
 * errors as for the calls it makes.  The plan lives only inside the call (the descriptor upload stages
 * it out of host memory before returning). */
sp_status sp_run_pass(const sp_shape* shape, int32_t n_branches, const int32_t* req_of_branch,
                      const int64_t* tok_offsets, const int32_t* tokens, int64_t node_rows,
                      const void* q, const void* k, const void* v, void* kv_pool,
                      int32_t pool_pages, void* out, float* lse, void* desc, size_t desc_bytes,
                      void* attn_ws, size_t attn_ws_bytes, const void* h, const void* W,
                      const int32_t* label_off, const int32_t* label_ids, int32_t n_labels,
                      float* logprobs, float* lse_vocab, void* lm_ws, size_t lm_ws_bytes,
                      float* probs, int32_t* argmax, void* stream, sp_plan_stats* stats);

/* One device input set of sp_run_pass_host, owned by the caller: device
 * buffers the pass's inputs are copied into, a pinned host buffer the launch
 * descriptor is staged in, and two CUDA events (cudaEvent_t, created by the
 * caller; timing may be disabled).  done_event is recorded on `stream` at the
 * end of every pass that used the set; copied_event on copy_stream once the
 * set's copies are done.  A caller alternates two sets so that one pass's
 * copies overlap the previous pass's kernels. */
typedef struct sp_input_set {
  void* q;               /* DEVICE bf16, q_rows rows of n_q_heads * head_dim   */
  void* k;               /* DEVICE bf16, q_rows rows of n_kv_heads * head_dim  */
  void* v;               /* DEVICE bf16, as k                                  */
  void* h;               /* DEVICE bf16, h_rows rows of hidden                 */
  int32_t* label_off;    /* DEVICE int32, h_rows + 1                           */
  int32_t* label_ids;    /* DEVICE int32, labels_cap                           */
  int64_t q_rows;
  int64_t h_rows;
  int64_t labels_cap;
  void* desc_host;       /* pinned HOST, desc_host_bytes                       */
  size_t desc_host_bytes;
  void* done_event;      /* cudaEvent_t                                        */
  void* copied_event;    /* cudaEvent_t                                        */
} sp_input_set;

/* sp_run_pass with its inputs and outputs in pinned host memory: the same
 * pass, plus the copies a caller holding host buffers needs, enqueued
 * without blocking on the pass's own work.
 *   1. plans and checks every capacity (as sp_run_pass; the set's q_rows,
 *      h_rows, labels_cap and desc_host_bytes too, SP_ERR_WORKSPACE) and the
 *      host label CSR (sp_check_labels, SP_ERR_ARG), before anything is
 *      enqueued;
 *   2. waits on the host for set->done_event: the last pass that used the
 *      set has finished, so its buffers and staging can be overwritten;
 *   3. on copy_stream: copies q_host, k_host, v_host (node_rows rows each),
 *      h_host (n_branches rows), label_off_host (n_branches + 1) and
 *      label_ids_host (n_labels) into the set, then uploads the descriptor
 *      from desc_host into desc (after any earlier sp_run_pass_host pass
 *      that reads the same desc buffer has finished: the library keeps one
 *      event per recently used desc buffer for this), then records
 *      copied_event;
 *   4. on stream: waits for copied_event, runs the tree attention, readout
 *      and softmax on the set's buffers, copies probs and argmax to
 *      probs_host and argmax_host, and records done_event.
 * The descriptor travels on copy_stream so that it reaches the copy engine
 * before the next call's input copies; on stream it would wait behind them
 * and the pass could not overlap the next call's copies.
 * Once step 3 has been enqueued, done_event is recorded even when a later
 * step fails.  The outputs in host memory are ready once done_event has
 * completed (or `stream` is synchronised).  All host buffers but tokens and
 * the CSRs must be pinned for the copies to run asynchronously; pageable
 * ones still work but their copies block the host.  Other arguments and
 * errors are as for sp_run_pass. */
sp_status sp_run_pass_host(const sp_shape* shape, int32_t n_branches,
                           const int32_t* req_of_branch, const int64_t* tok_offsets,
                           const int32_t* tokens, int64_t node_rows, const void* q_host,
                           const void* k_host, const void* v_host, const void* h_host,
                           const int32_t* label_off_host, const int32_t* label_ids_host,
                           int32_t n_labels, const sp_input_set* set, void* kv_pool,
                           int32_t pool_pages, void* out, float* lse, void* desc,
                           size_t desc_bytes, void* attn_ws, size_t attn_ws_bytes, const void* W,
                           float* logprobs, float* lse_vocab, void* lm_ws, size_t lm_ws_bytes,
                           float* probs, int32_t* argmax, float* probs_host,
                           int32_t* argmax_host, void* stream, void* copy_stream,
                           sp_plan_stats* stats);

/* Host-side validation of the option CSRs of sp_option_softmax (HOST
 * arrays): opt_off starts at 0, increases strictly and ends <= n_rows; q_off
 * starts at 0, ends <= n_opts, and gives every question 2..64 options.
 * SP_OK or SP_ERR_ARG. */
sp_status sp_check_options(const int32_t* opt_off, int32_t n_opts, int32_t n_rows,
                           const int32_t* q_off, int32_t n_questions);

/* Host-side validation of a label CSR (HOST arrays): counts in [2, 64],
 * 0 <= id < vocab, monotone offsets.  SP_OK or SP_ERR_ARG. */
sp_status sp_check_labels(const int32_t* label_off, const int32_t* label_ids, int32_t N,
                          int32_t vocab);

/* Bounded device wait on a flag, with the time limit and error path of
 * every pipeline wait inside libsp's kernels: one thread polls *flag until
 * it equals `expect` or limit_ns of device time (clamped to 1 us .. 2 s) has
 * passed.  On timeout it raises SP_ERR_DEVICE_TIMEOUT through the device
 * error word (read by sp_check_device_error) and returns; the context stays
 * usable.  For checking failure reporting without a fault: a flag that
 * nothing sets makes the wait run out.
 *   flag  DEVICE uint32, 4-byte aligned;  limit_ns >= 0 */
sp_status sp_wait_flag(const uint32_t* flag, uint32_t expect, int64_t limit_ns, void* stream);

/* Synchronise `stream`, read and clear the device error word of the current
 * device.  SP_OK, SP_ERR_DEVICE_TIMEOUT, SP_ERR_DEVICE_BOUNDS or SP_ERR_CUDA. */
sp_status sp_check_device_error(void* stream);

const char* sp_status_str(sp_status s);

/* Number of kernel launches the last attention / readout entry point
 * enqueued on this thread (for launch accounting). */
int32_t sp_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SP_H_ */
