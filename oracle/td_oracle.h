/*
 * td_oracle.h - plain, slow, single-threaded CPU definition of the collective KV path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or includes this
 * file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code with the CUDA path.
 *
 * Source of the method: "TokenDance: Scaling Multi-Agent LLM Serving via Collective KV
 * Cache Sharing" (arXiv 2604.03143), as described on the pages
 *   [R] zhaifeiyue.github.io/papers/2604.03143/detail.html (a structured review), and
 *   [B] the juhe.plus blog post on the same paper.
 * Citations below name the page and its section / figure / table.
 *
 * Every step is written in the order the method states it, on dense host arrays, without
 * blocking or fusion. Readings of points the pages leave open are marked READING.
 *
 * Layouts (all row-major, bf16 stored as its 16-bit pattern in uint16_t):
 *   canonical K/V        [L][S][E]           E = H*D, canonical token order
 *   paged pool           [L][2][num_pages][P][H][D]   (index 0 = K, 1 = V)
 *   block table          [N][max_lp] int32   logical page -> physical page, -1 unmapped
 *   fresh K (check)      [N][S][E]           agent frame, canonical token order
 *   fresh K/V (selected) [N][nl][k][E]       agent frame, row r = token sel[i][r]
 *   master K/V           [nl][S][E]          canonical frame, nl = layer_end - layer_begin
 *   store rows           [N][nl], CSR        rowptr [N*nl+1], block idx [nnz],
 *                                            values [nnz][B][E] (K and V)
 */
#ifndef TD_ORACLE_H
#define TD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_CAPACITY = 3, ORC_ERR_UNMAPPED = 4,
       ORC_ERR_NONFINITE = 5 };

typedef struct {
  int n_layers;    /* L */
  int n_kv_heads;  /* H */
  int head_dim;    /* D, multiple of 16 */
  int page_size;   /* P tokens per page */
  int diff_block;  /* B tokens per diff block, canonical axis */
  double rope_theta;
} orc_shape;

typedef struct {
  int n_agents;            /* N */
  int n_blocks;            /* M */
  const int32_t* block_len; /* [M] */
  const int32_t* hist_len;  /* [N] */
  const int32_t* perm;      /* [N*M]: perm[i*M+q] = block at slot q of agent i */
} orc_round;

typedef struct {
  uint16_t* base;          /* [L][2][num_pages][P][H][D] */
  int64_t num_pages;
  const int32_t* block_table; /* [N][max_lp] */
  int max_lp;
} orc_pool;

/* bf16 <-> float, round to nearest even, NaN kept quiet. */
float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);

/* Offsets of each shared block in each agent's prompt (Summary / Figure 1). */
int orc_offsets(const orc_round* rd, int32_t* off /* [N*M] */);

/* cos/sin of the RoPE angles at absolute offset a, frequencies f < D/2. */
void orc_rope_table(int64_t a, int head_dim, double theta, float* c, float* s);

/* Rotate one token row by the table (inverse = rotate by -a). */
void orc_rotate_row(const uint16_t* x, uint16_t* y, int n_heads, int head_dim,
                    const float* c, const float* s, int inverse);

/* The same rotation in float64 from bf16 inputs, no rounding of the result. */
void orc_rotate_row_f64(const uint16_t* x, double* y, int n_heads, int head_dim,
                        int64_t a, double theta, int inverse);

/* Stage 1: collective re-rotation of the shared blocks into every agent's pages. */
int orc_rerotate(const orc_shape* sh, const orc_round* rd, const uint16_t* k_canon,
                 const uint16_t* v_canon, int layer_begin, int layer_end, orc_pool* pool);

/* Squared key deviation of one token row, in the fixed summation order. */
float orc_token_dev(const uint16_t* fresh, const uint16_t* reused, int elems);

/* Stage 2: deviation at the check layer and per-agent top-k selection. */
int orc_check_select(const orc_shape* sh, const orc_round* rd, int check_layer,
                     const orc_pool* pool, const uint16_t* k_fresh, int recompute_pct,
                     int32_t* sel /* [N*k] */, float* dev /* [N*S] or NULL */, int* k_out);

/* Top-k of one agent's deviations: larger first, ties to the lower token; output ascending. */
int orc_topk(const float* dev, int n, int k, int32_t* out);

/* Stage 3a: master choice. cost [N] may be NULL. Returns the master index (or <0). */
int orc_pick_master(int n_agents, int n_shared, int diff_block, const int32_t* sel, int k,
                    int64_t* cost);

/* Stage 3a, variant: the agent whose selected tokens deviate least in total. score[i] =
 * sum over the k selected tokens of dev_i, in float64, in the fixed order of the variant
 * (see the source). Returns the master (or <0 on bad input / non-finite scores). */
int orc_pick_master_min_dev(int n_agents, int n_shared, const int32_t* sel, int k,
                            const float* dev, double* score);

/* Stage 2, variant: one important set for the whole group: the top-k tokens of the
 * group deviation g(t) = sum over agents of dev_i(t) (float32, agents in order). */
int orc_select_group(const float* dev, int n_agents, int n_shared, int k, int32_t* sel_row,
                     float* group_dev);

/* Stage 3b: Master-Mirror encoding of layers [layer_begin, layer_end). */
int orc_diff_encode(const orc_shape* sh, const orc_round* rd, int master,
                    const uint16_t* k_canon, const uint16_t* v_canon,
                    const int32_t* sel, int k,
                    const uint16_t* k_fresh_sel, const uint16_t* v_fresh_sel,
                    int layer_begin, int layer_end,
                    uint16_t* master_k, uint16_t* master_v,
                    int64_t* rowptr, int32_t* block_idx, uint16_t* val_k, uint16_t* val_v,
                    int64_t capacity, int64_t* nnz_out);

/* Stage 4: restore agents' paged KV from the Master and the diffs. frame 0 = agent frame
 * (RoPE recovered), 1 = canonical frame (plain copy). */
int orc_fused_restore(const orc_shape* sh, const orc_round* rd, int master,
                      const uint16_t* master_k, const uint16_t* master_v,
                      const int64_t* rowptr, const int32_t* block_idx,
                      const uint16_t* val_k, const uint16_t* val_v,
                      const int32_t* agents, int n_list, int layer_begin, int layer_end,
                      int frame, orc_pool* pool);

/* Decode attention of the listed agents read straight from the Master and the diffs
 * (no restored cache): history K/V from the pool, shared K = R(off) X_a, V = X_a; float64.
 * q [nl][n_list][n_q_heads][D] bf16, out [nl][n_list][n_q_heads][D], lse [nl][n_list][n_q_heads]
 * or NULL. The store holds exactly the layers [layer_begin, layer_end). from_pool != 0:
 * every position [0, h_a + S) from the pages instead (a restored cache). */
int orc_attention(const orc_shape* sh, const orc_round* rd, int master,
                  const uint16_t* master_k, const uint16_t* master_v,
                  const int64_t* rowptr, const int32_t* block_idx,
                  const uint16_t* val_k, const uint16_t* val_v, const orc_pool* pool,
                  const int32_t* agents, int n_list, int layer_begin, int layer_end,
                  const uint16_t* q, int n_q_heads, double scale, int from_pool, double* out,
                  double* lse);

/* Compression ratios (Performance Evaluation, metric "compression ratio"). */
double orc_round_ratio(int n_agents, int n_layers, int n_shared, int elems, int diff_block,
                       int64_t nnz);
double orc_mirror_ratio(int n_layers, int n_shared, int elems, int diff_block,
                        int64_t nnz_mirror);

#ifdef __cplusplus
}
#endif
#endif
