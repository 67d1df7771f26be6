/*
 * td.h - C ABI of the collective KV cache path on GB300 (sm_103a).
 *
 * The path is the data-parallel core of TokenDance ("TokenDance: Scaling Multi-Agent LLM
 * Serving via Collective KV Cache Sharing", arXiv 2604.03143), as described by the
 * structured review at zhaifeiyue.github.io/papers/2604.03143/detail.html (cited as [R])
 * and the juhe.plus blog post on the paper (cited as [B]). One All-Gather round: N agents
 * share M output blocks; agent i sees its private history H_i followed by the blocks in
 * its own order Pi_i ([R] Summary, Motivation; Figure 1). Four stages:
 *   1 td_rerotate_batched  one launch turns the shared blocks' canonical-frame K to every
 *                          agent's offsets and writes all agents' paged KV
 *   2 td_check_select      one key-deviation pass at the check layer picks each agent's
 *                          important (to be recomputed) positions
 *   3 td_pick_master       picks the Master agent;
 *     td_diff_encode       stores the Master dense and every other agent (Mirror) as
 *                          block-sparse K/V diffs
 *   4 td_fused_restore     gathers the Master, merges each agent's diffs, turns K back to
 *                          the agent's offsets and writes its paged KV; no dense Mirror
 *
 * Conventions for every call
 *   - Device pointers are CUDA device addresses of the current device; host pointers are
 *     ordinary host memory. Each argument says which it is. All memory is owned by the
 *     caller except the context's private workspace.
 *   - bf16 tensors are raw 16-bit patterns, row-major. E = n_kv_heads * head_dim.
 *   - S = sum of block_len (shared tokens). B = td_shape.diff_block tokens per diff block
 *     (16 or 32) and nb = ceil(S / B) diff blocks.
 *   - Calls are asynchronous on `stream` (a cudaStream_t) unless stated otherwise.
 *   - Concurrency on one context. A context is used by one host thread at a time. Its
 *     calls may be issued on several streams:
 *       . the round's tables (offsets, RoPE, token blocks) are the context's and shared:
 *         a stream's first call after they are uploaded is ordered after the upload, and
 *         a call with a different round waits on the device (events on the other streams,
 *         no host blocking) until every earlier call that reads the old tables has
 *         finished before it replaces them;
 *       . beyond the tables, calls of one group share scratch, so at most one call of
 *         each group may be in flight at a time (order them: one stream, or events):
 *           selection  td_check_select, td_check_select_group
 *           master     td_pick_master, td_pick_master_min_deviation
 *           encode     td_diff_encode
 *           attention  td_fused_attention, td_paged_attention
 *         td_rerotate_batched, td_fused_restore and td_materialise_mirror use no scratch.
 *       Calls of different groups may overlap: for example td_check_select and
 *       td_pick_master on one stream while td_rerotate_batched of other layers runs on
 *       another. Data the caller passes (pool, store, selection) is the caller's to order.
 *     Inside a stream capture nothing is tracked and a change of round is refused
 *     (TD_ERR_INVALID_ARG): make a call with the round, and let it finish, before
 *     capturing calls that use it.
 *   - Host validation runs first; an invalid argument returns TD_ERR_INVALID_ARG and
 *     launches nothing. A CUDA launch or copy failure returns TD_ERR_CUDA.
 *   - Faults found on the device never trap: the offending write is skipped and a bit
 *     is set in the context's error word, read and cleared by td_get_error.
 *   - Every output is a deterministic function of the inputs.
 */
#ifndef TD_H
#define TD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum td_status {
  TD_OK = 0,
  TD_ERR_INVALID_ARG = 1,    /* bad shape, pointer, range or size; nothing launched */
  TD_ERR_CUDA = 2,           /* a CUDA runtime call failed */
  TD_ERR_CAPACITY = 3,       /* diff store too small (see td_diff_encode) */
  TD_ERR_UNMAPPED_PAGE = 4,  /* a block-table entry was -1 or >= num_pages */
  TD_ERR_NONFINITE = 5,      /* a key deviation was NaN or infinite */
  TD_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait on its own copies ran out */
  TD_ERR_SCRATCH_LIMIT = 7   /* sizes exceed the fixed scratch of td_check_select_noalloc */
} td_status;

/* Model shape. head_dim must be a multiple of 16 (RoPE pairs element f with f + D/2 and
 * the kernels move 8 elements per 16-byte vector); diff_block is 16 or 32 (a 32-token diff
 * block is one 32-token page: the pages' "diff block = page size" reading). */
typedef struct td_shape {
  int32_t n_layers;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t page_size;    /* tokens per KV page, >= 1 */
  int32_t diff_block;   /* tokens per diff block on the canonical axis: 16 or 32 */
  double rope_theta;    /* RoPE base, e.g. 1e6 for Qwen2.5 */
} td_shape;

/* One All-Gather round ([R] Summary, Motivation: P_i = H_i || Pi_i(O); Figure 1).
 * All arrays are HOST memory, read during the call only. Block j's offset in agent i's
 * prompt is hist_len[i] plus the lengths of the blocks that perm[i] places before j. */
typedef struct td_round {
  int32_t n_agents;          /* N >= 1 */
  int32_t n_blocks;          /* M >= 1 */
  const int32_t* block_len;  /* [M] host, each >= 1 */
  const int32_t* hist_len;   /* [N] host, each >= 0 */
  const int32_t* perm;       /* [N*M] host; perm[i*M+q] = block at slot q of agent i */
} td_round;

/* Paged KV cache shared by all agents ([R] §3d, §5: vLLM paged KV with block tables).
 * base: DEVICE, bf16, layout [L][2][num_pages][page_size][H][D] (index 0 = K, 1 = V).
 * block_table: DEVICE int32 [N][max_pages_per_agent]; entry = physical page of the
 * agent's logical page, -1 = unmapped. The token at prompt position p of agent i lives in
 * page block_table[i][p / page_size], slot p % page_size. Only positions of the shared
 * span are written; pages holding only history may stay unmapped. */
typedef struct td_paged {
  void* base;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t max_pages_per_agent;
} td_paged;

/* Master-Mirror diff store ([R] Summary Method (3); Figure 8; §2b item 2: one
 * (indices, values) record per Mirror per layer). All pointers DEVICE, caller-allocated.
 * It covers the layers [layer_begin, layer_end) it was encoded for; nl = their count.
 * K is kept in the canonical frame (block-local RoPE positions).
 *   master_k, master_v  bf16 [nl][S][E]       the Master's cache, dense
 *   rowptr              int64 [N*nl + 1]      CSR rows, row = agent*nl + (layer-layer_begin)
 *   block_idx           int32 [capacity]      diff block index b of each record, ascending
 *                                             within a row
 *   val_k, val_v        bf16 [capacity][B][E] the Mirror's whole block; tokens past S are 0
 *   slot                int32 [N*nl*nb]       record of (agent, layer, block), or -1
 *   capacity_blocks     records the value arrays can hold
 * The Master's rows are empty. The arrays may also live in page-locked host memory that
 * the device addresses directly (cudaHostAlloc; on GB300 reached over NVLink-C2C): this
 * is the pages' storage tier ([R] §2a "Diff serialize ... GPU->CPU/Storage", "Fused
 * restore"), with encode writing and restore reading it in place. */
typedef struct td_diff_store {
  void* master_k;
  void* master_v;
  int64_t* rowptr;
  int32_t* block_idx;
  void* val_k;
  void* val_v;
  int32_t* slot;
  int64_t capacity_blocks;
  int32_t layer_begin;   /* written by td_diff_encode */
  int32_t layer_end;     /* written by td_diff_encode */
} td_diff_store;

typedef struct td_ctx td_ctx;

/* Create a context for one model shape. It owns only scratch space: the round's offset
 * and RoPE tables, the per-agent rank and mask tables, the deviations when the caller
 * does not keep them, the encode flags, and the error word. Limits: N <= max_agents,
 * M <= max_blocks, S <= max_shared. Uses the current CUDA device. Synchronous. */
td_status td_ctx_create(const td_shape* shape, int32_t max_agents, int32_t max_blocks,
                        int32_t max_shared, td_ctx** out);
td_status td_ctx_destroy(td_ctx* ctx);

/* Static text for a status code. */
const char* td_status_string(td_status s);

/* Block offsets of a round (host only): off_out[i*M + j] = prompt position where block j
 * starts in agent i ([R] Summary, Motivation; Figure 1). off_out: HOST int32 [N*M]. */
td_status td_round_offsets(const td_round* round, int32_t* off_out);

/* Stage 1 - collective re-rotation ([R] Summary Method (2): the round's requests are
 * batched and RoPE runs once for the group; Figure 7 T3; §2a "Collective prefill").
 * For every agent i, layer l in [layer_begin, layer_end) and shared token t of block j at
 * local index u: pool K of agent i at position off_ij + u = bf16(R(off_ij) Kc[l][t]) and,
 * when v_canon is not NULL, pool V there = Vc[l][t]. RoPE: neox pairing (f, f + D/2),
 * angle off * theta^(-2f/D), cos/sin computed in float64 on the host and rounded to float;
 * y0 = fma(x0, c, -(x1*s)), y1 = fma(x1, c, x0*s) in float32, rounded to bf16 (nearest
 * even). k_canon, v_canon: DEVICE bf16 [layer_end-layer_begin][S][E] (row 0 = layer
 * layer_begin). Canonical frame: block j's K rotated as if the block started at 0. */
td_status td_rerotate_batched(td_ctx* ctx, const td_round* round, const void* k_canon,
                              const void* v_canon, int32_t layer_begin, int32_t layer_end,
                              const td_paged* pool, void* stream);

/* Stage 2 - key deviation at the check layer and per-agent top-k ([R] Summary Method (2):
 * one key-difference analysis at the check layer, whose important positions all later
 * layers reuse; §3c A3). dev_i(t) = sum over the E elements of (fresh - reused)^2 in
 * float32, summed in a fixed order (16-byte vector v -> lane v mod 32, lanes ascending
 * through their vectors with fma, then a pairwise tree over the 32 lanes). reused = pool K
 * of agent i at its position of t, layer check_layer. k = ceil(recompute_pct * S / 100);
 * sel_i = the k tokens of largest dev (ties to the lower token), ascending.
 *   k_fresh  DEVICE bf16 [N][S][E]   recomputed K at the check layer, agent frame,
 *                                    canonical token order
 *   sel      DEVICE int32 [N][k]     output
 *   dev_out  DEVICE float [N][S]     output, or NULL
 *   k_out    HOST int32              k (computed on the host; no sync)
 * A non-finite deviation sets TD_ERR_NONFINITE in the error word (selection undefined). */
td_status td_check_select(td_ctx* ctx, const td_round* round, int32_t check_layer,
                          const td_paged* pool, const void* k_fresh, int32_t recompute_pct,
                          int32_t* sel, float* dev_out, int32_t* k_out, void* stream);

/* Stage 3a - Master choice ([R] Summary Method (3): keep the agent with the smallest
 * deviation dense; §3c A2: chosen by a deviation score so the diffs are sparsest).
 * mask_i = diff blocks (B tokens) holding a token of sel_i; cost(m) = sum over i != m of
 * |mask_i OR mask_m| (the number of diff blocks per layer the Mirrors can need);
 * master = argmin, ties to the lower index.
 *   sel          DEVICE int32 [N][k]
 *   cost_out     DEVICE int64 [N], or NULL
 *   master_dev   DEVICE int32, output (read by td_diff_encode)
 *   master_host  HOST int32, or NULL; when given the call synchronizes the stream */
td_status td_pick_master(td_ctx* ctx, const td_round* round, const int32_t* sel, int32_t k,
                         int64_t* cost_out, int32_t* master_dev, int32_t* master_host,
                         void* stream);

/* Stage 2, variant reading - one important set for the whole group. [R] Summary Method
 * (2) speaks of one key-difference analysis for the batched requests; this variant takes
 * it group-wide: the group deviation of token t is the float32 sum, in agent order, of
 * the agents' deviations (defined as for td_check_select), and its top k tokens (ties to
 * the lower token, ascending) become EVERY agent's selection: every row of sel is equal.
 *   group_dev_out  DEVICE float [S], or NULL
 * Other arguments as for td_check_select. */
td_status td_check_select_group(td_ctx* ctx, const td_round* round, int32_t check_layer,
                                const td_paged* pool, const void* k_fresh,
                                int32_t recompute_pct, int32_t* sel, float* dev_out,
                                float* group_dev_out, int32_t* k_out, void* stream);

/* Stage 3a, variant reading - the Master is "the agent with the smallest deviation"
 * ([R] Summary Method (3)) taken literally: score(i) = sum over i's k selected tokens of
 * dev_i(t), in float64, addend r to accumulator r mod 32 (ascending r), then the 32
 * accumulators added pairwise (l + 16, ..., l + 1); master = argmin, ties to the lower
 * index. A non-finite score sets TD_ERR_NONFINITE in the error word.
 *   dev        DEVICE float [N][S]  deviations as td_check_select writes them
 *   score_out  DEVICE double [N], or NULL
 * Other arguments as for td_pick_master. */
td_status td_pick_master_min_deviation(td_ctx* ctx, const td_round* round, const int32_t* sel,
                                       int32_t k, const float* dev, double* score_out,
                                       int32_t* master_dev, int32_t* master_host,
                                       void* stream);

/* Stage 3b - Master-Mirror block-sparse encoding ([R] Summary Method (3): Master keeps a
 * full cache, every other agent records only the indices and values of its differing
 * blocks; Figure 8; §2a "Diff serialize: Mirror dense -> (indices, K/V)"). Agent i's
 * canonical cache X_i(t) is its recomputed K turned back by R(-off) (same float32 / bf16
 * rounding as stage 1, with the signs of R(-a)) and recomputed V at t in sel_i, and the
 * canonical K/V elsewhere. The store receives X_master densely and, for each Mirror i,
 * layer and diff block b in ascending order, X_i's block b when any K or V bit of the
 * block differs from X_master's. No Mirror is ever materialised densely.
 *   master       DEVICE int32 (as written by td_pick_master, or the caller's choice)
 *   k_canon, v_canon   DEVICE bf16 [nl][S][E], row 0 = layer layer_begin
 *   sel          DEVICE int32 [N][k], each row ascending, as td_check_select writes it
 *   k_fresh_sel, v_fresh_sel  DEVICE bf16 [N][nl][k][E]: recomputed K (agent frame) and V
 *                of sel[i][r] at layer layer_begin + l in row [i][l][r]
 *   store        caller-allocated; capacity_blocks must be at least the candidate bound
 *                nl * cost(master) (cost as td_pick_master defines it), because blocks
 *                are first written at positions derived from the masks
 *   nnz_out      HOST int64, or NULL. When given, the call synchronizes the stream and
 *                returns TD_ERR_CAPACITY if the bound exceeds the capacity (then
 *                *nnz_out = the bound); otherwise *nnz_out = records written.
 * When the bound exceeds the capacity only master_k/master_v and rowptr are written and
 * TD_ERR_CAPACITY is also set in the error word. */
td_status td_diff_encode(td_ctx* ctx, const td_round* round, const int32_t* master,
                         const void* k_canon, const void* v_canon, const int32_t* sel,
                         int32_t k, const void* k_fresh_sel, const void* v_fresh_sel,
                         int32_t layer_begin, int32_t layer_end, td_diff_store* store,
                         int64_t* nnz_out, void* stream);

/* Stage 4 - fused diff restore ([R] Summary Method (3): on read-back the diffs are merged
 * into the Master's data in flight and RoPE is recovered, with no dense Mirror; §2a
 * "Fused restore: Master chunk + diff -> paged KV"; §3d). For each listed agent a, layer
 * l in [layer_begin, layer_end) (inside the store's range) and token t: source = a's
 * diff record for (l, t / B) if present, else the Master; pool K at a's position of t =
 * bf16(R(off) source K) when frame == 0, or source K unchanged when frame == 1; pool V =
 * source V. Rounding as in stage 1.
 *   agents  HOST int32 [n_list], each in [0, N) */
td_status td_fused_restore(td_ctx* ctx, const td_round* round, const td_diff_store* store,
                           const int32_t* agents, int32_t n_list, int32_t layer_begin,
                           int32_t layer_end, int32_t frame, const td_paged* pool,
                           void* stream);

/* td_check_select without a context and without any device allocation. The paper has
 * no counterpart: this entry point exists for callers that may not call cudaMalloc (for
 * instance code that runs under a pool allocator that forbids it, or inside a process
 * whose device footprint must stay fixed after start-up). It computes exactly what
 * td_check_select computes (same kernels, same order of summation, same selection).
 * Its scratch - a copy of the round descriptor, the offset and token tables, the N*S
 * deviations and an error word - is one fixed array in device memory (about 4.5 MiB),
 * held by every GPU that loads the library until the process exits.
 * Limits: N <= 256, M <= 256, N*M <= 16384, S <= 65536, N*S <= 1048576; larger rounds
 * return TD_ERR_SCRATCH_LIMIT before anything is launched. diff_block may be 16 or 32 (the
 * selection does not depend on it).
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture. After a
 * device reset the next call looks the address up again (the device has a new context).
 * The round's host arrays are copied to the array on `stream`: when they are page-locked
 * the copy may run after the call returns, so keep them unchanged until the stream has
 * passed the call (pageable arrays are read before the call returns). Every call
 * reuses the same array: calls whose work can overlap on the GPU (different streams
 * without ordering between them, or several host threads) race on it and must be
 * serialized by the caller. The error word is cleared at the start of each call.
 *   shape, round  HOST, as for td_ctx_create / td_check_select
 *   pool, k_fresh, sel, k_out, check_layer, recompute_pct   as for td_check_select
 *   err_bits_out  HOST, or NULL; when given the call synchronizes the stream, stores the
 *                 device error word there and returns the lowest error code recorded */
td_status td_check_select_noalloc(const td_shape* shape, const td_round* round,
                                  int32_t check_layer, const td_paged* pool,
                                  const void* k_fresh, int32_t recompute_pct, int32_t* sel,
                                  int32_t* k_out, uint32_t* err_bits_out, void* stream);

/* Decode attention read straight from the Master and the diffs: the restore fused into
 * attention ([B] §4.4 "Fused Diff Restore": diffs applied block by block on chip, attention
 * right after, no materialised cache; [R] §8 open questions and §9). For every listed agent
 * a, layer l in [layer_begin, layer_end) and query head g: the context is a's private
 * history (positions [0, h_a), K/V read from the pages as stored; those pages must be
 * mapped) and its shared tokens (the Master's rows with a's records over them, in the
 * canonical frame): the shared token of block j at local index u has position off_aj + u,
 * K = R(off_aj) X and V = X. The pages of the shared span are not read.
 *   out[l][x][g] = sum_p softmax_p(scale * q[l][x][g] . K_p) V_p over the context
 *   lse[l][x][g] = ln sum_p exp(scale * q[l][x][g] . K_p)
 * Query head g reads kv head g / (n_q_heads / H) (grouped queries, at most 8 per kv head).
 * The kernel turns the query by R(-off_aj) once per block instead of turning keys.
 * Arithmetic: scores in float32 (a turned query split into two bf16 parts on the tensor
 * cores: 16 bits of the query kept), softmax and the weighted sum of V in float32.
 *   store     the round's Master-Mirror store; [layer_begin, layer_end) within its layers
 *   pool      the agents' pages (history), as for td_fused_restore
 *   agents    HOST [n_list] agent indices
 *   q         DEVICE bf16 [layer_end-layer_begin][n_list][n_q_heads][D], agent frame (rotated
 *             at the query's position), 4-byte aligned
 *   out       DEVICE float [layer_end-layer_begin][n_list][n_q_heads][D]
 *   lse       DEVICE float [layer_end-layer_begin][n_list][n_q_heads], or NULL
 * Head dims 64 and 128 (else TD_ERR_INVALID_ARG). The store must be in device memory (a
 * store kept in host memory is refused with TD_ERR_INVALID_ARG: restore from it instead).
 * The context owns the partial results' scratch and grows it when a call needs more (synchronising the stream first). An
 * unmapped history page sets TD_ERR_UNMAPPED_PAGE in the error word; a bounded wait on the
 * copy engine that runs out sets TD_ERR_DEVICE_TIMEOUT (that unit's result is not written). */
td_status td_fused_attention(td_ctx* ctx, const td_round* round, const td_diff_store* store,
                             const td_paged* pool, const int32_t* agents, int32_t n_list,
                             int32_t layer_begin, int32_t layer_end, const void* q,
                             int32_t n_q_heads, float scale, float* out, float* lse,
                             void* stream);

/* Comparison baseline, not on the path: the same decode attention over a restored cache,
 * every position [0, h_a + S) read from the agent's pages (after td_fused_restore, frame
 * 0): the unfused "restore, then attend" the pages compare against. Arguments and
 * arithmetic as td_fused_attention (queries used as given, no turning). */
td_status td_paged_attention(td_ctx* ctx, const td_round* round, const td_paged* pool,
                             const int32_t* agents, int32_t n_list, int32_t layer_begin,
                             int32_t layer_end, const void* q, int32_t n_q_heads, float scale,
                             float* out, float* lse, void* stream);

/* Comparison baseline, not on the path: the dense restore that td_fused_restore replaces
 * ([R] §3d and Figure 5: materialise the Mirror, then copy it into pages). Writes agent's
 * canonical-frame cache X_agent for layers [layer_begin, layer_end): the Master's rows
 * with the agent's records laid over them (the Master itself: the Master's rows).
 * dense_k, dense_v: DEVICE bf16 [layer_end-layer_begin][S][E], caller-owned, 16-byte
 * aligned. Following it with td_rerotate_batched of a one-agent round (the agent's
 * history and order, its block-table row) reproduces td_fused_restore's frame-0 pages.
 * A slot map entry beyond the store's capacity sets TD_ERR_INVALID_ARG in the error word
 * and leaves that block unwritten. */
td_status td_materialise_mirror(td_ctx* ctx, const td_round* round, const td_diff_store* store,
                                int32_t agent, int32_t layer_begin, int32_t layer_end,
                                void* dense_k, void* dense_v, void* stream);

/* ---- Round-aware prompts and the KV Collector (host only) --------------------------
 * [R] Summary Method (1): the application puts a reserved separator token ([B] §4.1:
 * <TTSEP>) in front of every shared output block, so the runtime can hash segments by
 * content and recognise the blocks agents share; Method (2) and §5 "Batch formation": the
 * KV Collector groups a round's requests that share the same active prompt length, the
 * same cached span and disjoint slot mappings, and falls back to per-request processing
 * for the rest. A prompt is [private history][SEP block][SEP block]...: the tokens before
 * the first separator are the history; each later segment starts at a separator, which
 * belongs to it (block lengths tile the prompt). Two blocks are the same block when their
 * tokens are equal (the hash only indexes; equality is checked on the tokens). */
typedef struct td_prompt {
  const int32_t* tokens;   /* HOST [n_tokens] */
  int64_t n_tokens;
  const int32_t* pages;    /* HOST physical page of each logical page of the prompt
                              ([ceil(n_tokens / page_size)]), or NULL */
} td_prompt;

typedef enum td_round_status {
  TD_ROUND_OK = 0,              /* joined a collective round */
  TD_ROUND_NO_BLOCKS = 1,       /* no separator: nothing shared; runs alone */
  TD_ROUND_REPEATED_BLOCK = 2,  /* the same block twice: not a round; runs alone */
  TD_ROUND_NOT_CACHED = 3       /* a block without cached canonical K/V; runs alone */
} td_round_status;

/* 64-bit FNV-1a over the little-endian bytes of the tokens (the segment index key). */
uint64_t td_segment_hash(const int32_t* tokens, int64_t n_tokens);

/* Group requests into collective rounds, in arrival order. A request with at least one
 * block, no block twice and (when cached_hashes is given) every block's td_segment_hash in
 * cached_hashes joins the first group with exactly its set of blocks none of whose members
 * uses a page that the request's shared span uses (pages given); otherwise it opens a new
 * group. Other requests get a group of their own and a fallback status. Groups are
 * numbered in order of their first member.
 *   prompts        HOST [n_prompts]
 *   cached_hashes  HOST [n_cached], or NULL: every block counts as cached
 *   group_of, status_of  HOST int32 [n_prompts], outputs; n_groups_out HOST int32 */
td_status td_form_rounds(const td_prompt* prompts, int32_t n_prompts, int32_t sep_token,
                         int32_t page_size, const uint64_t* cached_hashes, int32_t n_cached,
                         int32_t* group_of, int32_t* status_of, int32_t* n_groups_out);

/* The round descriptor of one group: members in arrival order, blocks in the order of
 * the first member's prompt, each member's history length and permutation (slot q of
 * member x holds block perm[x*M + q]) - ready for td_round. All HOST; capacities in
 * members and blocks; TD_ERR_CAPACITY when they are too small, TD_ERR_INVALID_ARG when
 * the group's members do not hold one same set of distinct blocks. */
td_status td_group_round(const td_prompt* prompts, int32_t n_prompts, int32_t sep_token,
                         const int32_t* group_of, int32_t group, int32_t cap_members,
                         int32_t cap_blocks, int32_t* members, int32_t* n_members,
                         int32_t* block_len, int32_t* n_blocks, int32_t* hist_len,
                         int32_t* perm);

/* Fault injection for tests; no counterpart in the paper. With bytes > 0 every later
 * td_fused_attention / td_paged_attention call on this context makes each stage's barrier
 * expect `bytes` more than its copies deliver, so every bounded wait runs out (0.2 s of
 * device time each): the units record TD_ERR_DEVICE_TIMEOUT in the error word, wait
 * (bounded) for their own copies and return, and the outputs are not valid. No copy is
 * lost and nothing faults: the context stays usable. bytes = 0 restores normal calls. */
td_status td_inject_attention_wait_fault(td_ctx* ctx, uint32_t bytes);

/* Synchronize the stream, read and clear the error word. Returns TD_OK when no device
 * fault was recorded, else the lowest td_status code recorded; bits_out (HOST, or NULL)
 * receives the whole word (bit c set = code c recorded). */
td_status td_get_error(td_ctx* ctx, void* stream, uint32_t* bits_out);

#ifdef __cplusplus
}
#endif
#endif /* TD_H */
