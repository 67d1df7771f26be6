/*
 * td_oracle.c - the CPU definition of the collective KV path (see td_oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: the plain, slow reference the CUDA path is checked against.
 * Compile with -ffp-contract=off so that every float expression rounds where written.
 */
#include "td_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 storage */
float orc_bf16_to_f32(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((b >> 16) | 0x40u); /* NaN */
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

/* ------------------------------------------------------------------ round structure */
/* [R] Summary, Motivation, and Figure 1: agent i's prompt is its private history H_i
 * followed by the shared output blocks in the order Pi_i, so block j starts at
 * |H_i| + (lengths of the blocks that Pi_i places before j). Separators take no
 * positions (READING: a caller that keeps them folds them into the block lengths). */
int orc_offsets(const orc_round* rd, int32_t* off) {
  int N = rd->n_agents, M = rd->n_blocks;
  for (int i = 0; i < N; ++i) {
    int64_t pos = rd->hist_len[i];
    for (int q = 0; q < M; ++q) {
      int j = rd->perm[(int64_t)i * M + q];
      if (j < 0 || j >= M) return ORC_ERR_ARG;
      off[(int64_t)i * M + j] = (int32_t)pos;
      pos += rd->block_len[j];
    }
  }
  return ORC_OK;
}

/* canonical start of every block and the block of every canonical token */
static void canon_layout(const orc_round* rd, int64_t* start, int32_t* tok_block) {
  int64_t s = 0;
  for (int j = 0; j < rd->n_blocks; ++j) {
    start[j] = s;
    for (int u = 0; u < rd->block_len[j]; ++u) tok_block[s + u] = j;
    s += rd->block_len[j];
  }
}

static int shared_len(const orc_round* rd) {
  int s = 0;
  for (int j = 0; j < rd->n_blocks; ++j) s += rd->block_len[j];
  return s;
}

/* ------------------------------------------------------------------ RoPE */
/* RoPE with the neox pairing used by Qwen2.5: element f of a head pairs with f + D/2 and
 * turns at angle a * theta^(-2f/D). [R] Deep Analysis §0 (the method relies on RoPE being
 * invertible) and §3e; [B] §3 (position-independent reuse works through RoPE).
 * READING (the pages give no arithmetic): cos and sin come from the float64 library
 * functions, rounded once to float; the angle is (double)a * pow(theta, -2f/D). */
void orc_rope_table(int64_t a, int head_dim, double theta, float* c, float* s) {
  for (int f = 0; f < head_dim / 2; ++f) {
    double inv_freq = pow(theta, -(double)(2 * f) / (double)head_dim);
    double ang = (double)a * inv_freq;
    c[f] = (float)cos(ang);
    s[f] = (float)sin(ang);
  }
}

/* READING of the rounding: each cross product x*s is rounded to float, then one fused
 * multiply-add forms the output, which is rounded to bf16 (nearest even).
 *   forward  R(+a): y0 = x0*c - x1*s,  y1 = x1*c + x0*s
 *   inverse  R(-a): y0 = x0*c + x1*s,  y1 = x1*c - x0*s                                  */
void orc_rotate_row(const uint16_t* x, uint16_t* y, int n_heads, int head_dim,
                    const float* c, const float* s, int inverse) {
  int half = head_dim / 2;
  for (int h = 0; h < n_heads; ++h) {
    const uint16_t* xh = x + (int64_t)h * head_dim;
    uint16_t* yh = y + (int64_t)h * head_dim;
    for (int f = 0; f < half; ++f) {
      float x0 = orc_bf16_to_f32(xh[f]);
      float x1 = orc_bf16_to_f32(xh[f + half]);
      float x1s = x1 * s[f];
      float x0s = x0 * s[f];
      float y0, y1;
      if (!inverse) {
        y0 = fmaf(x0, c[f], -x1s);
        y1 = fmaf(x1, c[f], x0s);
      } else {
        y0 = fmaf(x0, c[f], x1s);
        y1 = fmaf(x1, c[f], -x0s);
      }
      yh[f] = orc_f32_to_bf16(y0);
      yh[f + half] = orc_f32_to_bf16(y1);
    }
  }
}

void orc_rotate_row_f64(const uint16_t* x, double* y, int n_heads, int head_dim, int64_t a,
                        double theta, int inverse) {
  int half = head_dim / 2;
  double sign = inverse ? -1.0 : 1.0;
  for (int h = 0; h < n_heads; ++h) {
    for (int f = 0; f < half; ++f) {
      double ang = sign * (double)a * pow(theta, -(double)(2 * f) / (double)head_dim);
      double x0 = orc_bf16_to_f32(x[(int64_t)h * head_dim + f]);
      double x1 = orc_bf16_to_f32(x[(int64_t)h * head_dim + f + half]);
      y[(int64_t)h * head_dim + f] = x0 * cos(ang) - x1 * sin(ang);
      y[(int64_t)h * head_dim + f + half] = x1 * cos(ang) + x0 * sin(ang);
    }
  }
}

/* ------------------------------------------------------------------ paged pool */
/* Paged KV (vLLM-style, [R] §3d and §5 "Memory management"): the token at prompt
 * position p of agent i sits in physical page block_table[i][p / P], slot p % P. */
static uint16_t* pool_row(const orc_shape* sh, const orc_pool* pool, int agent, int layer,
                          int kv, int64_t pos, int* err) {
  int P = sh->page_size;
  int64_t lp = pos / P;
  if (lp >= pool->max_lp) { *err = ORC_ERR_UNMAPPED; return NULL; }
  int32_t page = pool->block_table[(int64_t)agent * pool->max_lp + lp];
  if (page < 0 || page >= pool->num_pages) { *err = ORC_ERR_UNMAPPED; return NULL; }
  int64_t E = (int64_t)sh->n_kv_heads * sh->head_dim;
  int64_t idx = ((((int64_t)layer * 2 + kv) * pool->num_pages + page) * P + pos % P) * E;
  return pool->base + idx;
}

/* ------------------------------------------------------------------ stage 1 */
/* Collective position-independent reuse. [R] Summary, Method (2): the N requests of a
 * round are batched and RoPE is applied once for the group; Figure 7 (T3) draws one RoPE
 * for all agents; §2a "Collective prefill ... [N, L, H, D] batched".
 * READING of the canonical frame ([B] §6 says the pages leave the RoPE-offset variant
 * open): block j's K is stored as if the block started at position 0, so agent i needs
 * R(off_ij) applied; V carries no position and is copied unchanged. */
int orc_rerotate(const orc_shape* sh, const orc_round* rd, const uint16_t* k_canon,
                 const uint16_t* v_canon, int layer_begin, int layer_end, orc_pool* pool) {
  int N = rd->n_agents, M = rd->n_blocks, H = sh->n_kv_heads, D = sh->head_dim;
  int64_t E = (int64_t)H * D;
  int S = shared_len(rd);
  int32_t* off = malloc(sizeof(int32_t) * N * M);
  int64_t* start = malloc(sizeof(int64_t) * (M + 1));
  int32_t* tok_block = malloc(sizeof(int32_t) * (S + 1));
  float* c = malloc(sizeof(float) * D);
  float* s = malloc(sizeof(float) * D);
  int status = orc_offsets(rd, off);
  canon_layout(rd, start, tok_block);
  for (int i = 0; i < N && status == ORC_OK; ++i) {
    for (int j = 0; j < M; ++j) {
      int32_t a = off[(int64_t)i * M + j];
      orc_rope_table(a, D, sh->rope_theta, c, s);
      for (int u = 0; u < rd->block_len[j]; ++u) {
        int64_t t = start[j] + u;
        for (int l = layer_begin; l < layer_end; ++l) {
          int err = ORC_OK;
          uint16_t* kdst = pool_row(sh, pool, i, l, 0, (int64_t)a + u, &err);
          if (!kdst) { status = err; continue; }
          orc_rotate_row(k_canon + ((int64_t)l * S + t) * E, kdst, H, D, c, s, 0);
          if (v_canon) {
            uint16_t* vdst = pool_row(sh, pool, i, l, 1, (int64_t)a + u, &err);
            memcpy(vdst, v_canon + ((int64_t)l * S + t) * E, sizeof(uint16_t) * E);
          }
        }
      }
    }
  }
  free(off); free(start); free(tok_block); free(c); free(s);
  return status;
}

/* ------------------------------------------------------------------ stage 2 */
/* Key deviation of one token: [R] Summary, Method (2) "one key-difference analysis at the
 * check layer"; Figure 7. READING: the squared L2 distance over all H*D elements of the
 * token, summed in float32 in this fixed order: the row is cut into 16-byte vectors of 8
 * elements; vector v goes to accumulator v mod 32; each accumulator takes its vectors in
 * ascending order and its elements in ascending order, acc = fma(d, d, acc), d = a - b;
 * the 32 accumulators are then added pairwise (l + 16, l + 8, l + 4, l + 2, l + 1). */
float orc_token_dev(const uint16_t* fresh, const uint16_t* reused, int elems) {
  float acc[32];
  for (int l = 0; l < 32; ++l) acc[l] = 0.0f;
  for (int v = 0; v < elems / 8; ++v) {
    int l = v % 32;
    for (int e = 8 * v; e < 8 * v + 8; ++e) {
      float d = orc_bf16_to_f32(fresh[e]) - orc_bf16_to_f32(reused[e]);
      acc[l] = fmaf(d, d, acc[l]);
    }
  }
  for (int w = 16; w >= 1; w /= 2)
    for (int l = 0; l < w; ++l) acc[l] = acc[l] + acc[l + w];
  return acc[0];
}

typedef struct { float dev; int32_t t; } dev_item;

static int cmp_dev_desc(const void* pa, const void* pb) {
  const dev_item* a = pa;
  const dev_item* b = pb;
  if (a->dev > b->dev) return -1;
  if (a->dev < b->dev) return 1;
  return (a->t > b->t) - (a->t < b->t);
}

static int cmp_i32(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* Important positions: the k tokens with the largest deviation ([R] Summary Method (2);
 * §3c A3: the set chosen at the check layer is reused by every later layer).
 * READING: ties go to the lower token index; the output is sorted ascending. */
int orc_topk(const float* dev, int n, int k, int32_t* out) {
  if (k < 0 || k > n) return ORC_ERR_ARG;
  dev_item* items = malloc(sizeof(dev_item) * (n > 0 ? n : 1));
  int status = ORC_OK;
  for (int t = 0; t < n; ++t) {
    if (isnan(dev[t]) || isinf(dev[t])) status = ORC_ERR_NONFINITE;
    items[t].dev = dev[t];
    items[t].t = t;
  }
  if (status == ORC_OK) {
    qsort(items, n, sizeof(dev_item), cmp_dev_desc);
    for (int r = 0; r < k; ++r) out[r] = items[r].t;
    qsort(out, k, sizeof(int32_t), cmp_i32);
  }
  free(items);
  return status;
}

/* READING of the fraction: k = ceil(pct * S / 100) of the S shared tokens, per agent. */
int orc_check_select(const orc_shape* sh, const orc_round* rd, int check_layer,
                     const orc_pool* pool, const uint16_t* k_fresh, int recompute_pct,
                     int32_t* sel, float* dev, int* k_out) {
  int N = rd->n_agents, M = rd->n_blocks;
  int64_t E = (int64_t)sh->n_kv_heads * sh->head_dim;
  int S = shared_len(rd);
  if (recompute_pct < 0 || recompute_pct > 100) return ORC_ERR_ARG;
  int k = (recompute_pct * S + 99) / 100;
  *k_out = k;
  int32_t* off = malloc(sizeof(int32_t) * N * M);
  int64_t* start = malloc(sizeof(int64_t) * (M + 1));
  int32_t* tok_block = malloc(sizeof(int32_t) * (S + 1));
  float* d = malloc(sizeof(float) * (S > 0 ? S : 1));
  int status = orc_offsets(rd, off);
  canon_layout(rd, start, tok_block);
  for (int i = 0; i < N && status == ORC_OK; ++i) {
    for (int t = 0; t < S; ++t) {
      int j = tok_block[t];
      int64_t pos = off[(int64_t)i * M + j] + (t - start[j]);
      int err = ORC_OK;
      const uint16_t* reused = pool_row(sh, pool, i, check_layer, 0, pos, &err);
      if (!reused) { status = err; break; }
      d[t] = orc_token_dev(k_fresh + ((int64_t)i * S + t) * E, reused, (int)E);
      if (dev) dev[(int64_t)i * S + t] = d[t];
    }
    if (status == ORC_OK) status = orc_topk(d, S, k, sel + (int64_t)i * k);
  }
  free(off); free(start); free(tok_block); free(d);
  return status;
}

/* ------------------------------------------------------------------ stage 3a */
/* Master choice: [R] Summary Method (3) keeps the agent "with the smallest deviation" as
 * the dense Master; §3c A2 says the choice is made by a deviation score so that the
 * diffs come out sparsest, and Figure 8 says the store consumes the reuse plan.
 * READING: the score of candidate m is the number of diff blocks its Mirrors can need,
 * sum over i != m of |mask_i OR mask_m|, where mask_i marks the B-token blocks that hold
 * a selected token of agent i; the smallest score wins, ties to the lower index. */
int orc_pick_master(int n_agents, int n_shared, int diff_block, const int32_t* sel, int k,
                    int64_t* cost) {
  int nb = (n_shared + diff_block - 1) / diff_block;
  unsigned char* mask = calloc((size_t)n_agents * (nb > 0 ? nb : 1), 1);
  for (int i = 0; i < n_agents; ++i)
    for (int r = 0; r < k; ++r) {
      int t = sel[(int64_t)i * k + r];
      if (t < 0 || t >= n_shared) { free(mask); return -ORC_ERR_ARG; }
      mask[(int64_t)i * nb + t / diff_block] = 1;
    }
  int best = -1;
  int64_t best_cost = 0;
  for (int m = 0; m < n_agents; ++m) {
    int64_t c = 0;
    for (int i = 0; i < n_agents; ++i) {
      if (i == m) continue;
      for (int b = 0; b < nb; ++b)
        c += (mask[(int64_t)i * nb + b] | mask[(int64_t)m * nb + b]) ? 1 : 0;
    }
    if (cost) cost[m] = c;
    if (best < 0 || c < best_cost) { best = m; best_cost = c; }
  }
  free(mask);
  return best;
}

/* Variant of the Master rule read literally: "the agent with the smallest deviation"
 * ([R] Summary, Method (3)) taken as the total key deviation of the agent's important
 * positions. READING of the summation: float64; addend r goes to accumulator r mod 32,
 * each accumulator adds its addends in ascending r, then the 32 accumulators are added
 * pairwise (l + 16, l + 8, ..., l + 1). Smallest score wins, ties to the lower index. */
int orc_pick_master_min_dev(int n_agents, int n_shared, const int32_t* sel, int k,
                            const float* dev, double* score) {
  int best = -1;
  double best_score = 0.0;
  for (int i = 0; i < n_agents; ++i) {
    double acc[32];
    for (int l = 0; l < 32; ++l) acc[l] = 0.0;
    for (int r = 0; r < k; ++r) {
      int t = sel[(int64_t)i * k + r];
      if (t < 0 || t >= n_shared) return -ORC_ERR_ARG;
      acc[r % 32] = acc[r % 32] + (double)dev[(int64_t)i * n_shared + t];
    }
    for (int w = 16; w >= 1; w /= 2)
      for (int l = 0; l < w; ++l) acc[l] = acc[l] + acc[l + w];
    if (isnan(acc[0]) || isinf(acc[0])) return -ORC_ERR_NONFINITE;
    if (score) score[i] = acc[0];
    if (best < 0 || acc[0] < best_score) { best = i; best_score = acc[0]; }
  }
  return best;
}

/* Variant of the important-position set: one set for the whole group ([R] Summary,
 * Method (2): one key-difference analysis for the batch of N requests). READING: the
 * group deviation of token t is the float32 sum of the agents' deviations in agent order
 * 0..N-1; the top-k of it (ties to the lower token, ascending output) is every agent's
 * set. */
int orc_select_group(const float* dev, int n_agents, int n_shared, int k, int32_t* sel_row,
                     float* group_dev) {
  float* g = malloc(sizeof(float) * (n_shared > 0 ? n_shared : 1));
  for (int t = 0; t < n_shared; ++t) {
    float s = 0.0f;
    for (int i = 0; i < n_agents; ++i) s = s + dev[(int64_t)i * n_shared + t];
    g[t] = s;
    if (group_dev) group_dev[t] = s;
  }
  int st = orc_topk(g, n_shared, k, sel_row);
  free(g);
  return st;
}

/* ------------------------------------------------------------------ stage 3b */
/* Agent i's cache in the canonical frame at layer l (dense, one layer): the recomputed
 * K/V at its selected tokens, K turned back by R(-off), and the reused canonical K/V
 * everywhere else. [R] Summary Method (2): selective recompute refreshes the important
 * positions; Method (3) stores Master and Mirrors; READING: the store keeps the
 * canonical frame so Master and Mirrors can be compared without positions. */
static void build_agent_cache(const orc_shape* sh, int S, int M, const int32_t* off_i,
                              const int32_t* tok_block, const uint16_t* kc_l,
                              const uint16_t* vc_l, const int32_t* sel_i, int k,
                              const uint16_t* kf_il, const uint16_t* vf_il, uint16_t* xk,
                              uint16_t* xv, float* c, float* s) {
  int H = sh->n_kv_heads, D = sh->head_dim;
  int64_t E = (int64_t)H * D;
  (void)M;
  memcpy(xk, kc_l, sizeof(uint16_t) * S * E);
  memcpy(xv, vc_l, sizeof(uint16_t) * S * E);
  for (int r = 0; r < k; ++r) {
    int t = sel_i[r];
    orc_rope_table(off_i[tok_block[t]], D, sh->rope_theta, c, s);
    orc_rotate_row(kf_il + (int64_t)r * E, xk + (int64_t)t * E, H, D, c, s, 1);
    memcpy(xv + (int64_t)t * E, vf_il + (int64_t)r * E, sizeof(uint16_t) * E);
  }
}

/* Master-Mirror diff: [R] Summary Method (3): the Master keeps its full cache and every
 * other agent is a block-sparse K/V diff that records only the indices and values of the
 * differing blocks; Figure 8 "Diff = block-sparse (indices, values)"; §2a "Diff
 * serialize: Mirror dense -> (indices, K/V)"; §2b item 2: one (indices, values) record
 * per Mirror per layer. READING: K and V share one index list; a block is recorded when
 * any bit of its K or V differs from the Master's; the recorded values are the Mirror's
 * whole block; a tail block shorter than B is zero-padded. Rows run (agent asc, layer
 * asc) and indices ascend within a row; the Master's own rows are empty. */
int orc_diff_encode(const orc_shape* sh, const orc_round* rd, int master,
                    const uint16_t* k_canon, const uint16_t* v_canon, const int32_t* sel,
                    int k, const uint16_t* k_fresh_sel, const uint16_t* v_fresh_sel,
                    int layer_begin, int layer_end, uint16_t* master_k, uint16_t* master_v,
                    int64_t* rowptr, int32_t* block_idx, uint16_t* val_k, uint16_t* val_v,
                    int64_t capacity, int64_t* nnz_out) {
  int N = rd->n_agents, M = rd->n_blocks, B = sh->diff_block, D = sh->head_dim;
  int64_t E = (int64_t)sh->n_kv_heads * D;
  int S = shared_len(rd);
  int nl = layer_end - layer_begin;
  int nb = (S + B - 1) / B;
  if (master < 0 || master >= N || nl < 0) return ORC_ERR_ARG;
  int32_t* off = malloc(sizeof(int32_t) * N * M);
  int64_t* start = malloc(sizeof(int64_t) * (M + 1));
  int32_t* tok_block = malloc(sizeof(int32_t) * (S + 1));
  float* c = malloc(sizeof(float) * D);
  float* s = malloc(sizeof(float) * D);
  uint16_t* xik = malloc(sizeof(uint16_t) * ((int64_t)S * E + 1));
  uint16_t* xiv = malloc(sizeof(uint16_t) * ((int64_t)S * E + 1));
  int status = orc_offsets(rd, off);
  canon_layout(rd, start, tok_block);
  int64_t nnz = 0;

  /* the Master's own cache, stored dense */
  for (int li = 0; li < nl && status == ORC_OK; ++li) {
    int l = layer_begin + li;
    build_agent_cache(sh, S, M, off + (int64_t)master * M, tok_block,
                      k_canon + (int64_t)l * S * E, v_canon + (int64_t)l * S * E,
                      sel + (int64_t)master * k, k,
                      k_fresh_sel + (((int64_t)master * nl + li) * k) * E,
                      v_fresh_sel + (((int64_t)master * nl + li) * k) * E,
                      master_k + (int64_t)li * S * E, master_v + (int64_t)li * S * E, c, s);
  }

  /* every Mirror against it; count first so that an undersized store receives no values */
  for (int pass = 0; pass < 2 && status == ORC_OK; ++pass) {
    int write = pass == 1;
    if (write && nnz > capacity) { status = ORC_ERR_CAPACITY; break; }
    nnz = 0;
    for (int i = 0; i < N; ++i) {
      for (int li = 0; li < nl; ++li) {
        int l = layer_begin + li;
        if (write) rowptr[(int64_t)i * nl + li] = nnz;
        if (i == master) continue;
        const uint16_t* xmk = master_k + (int64_t)li * S * E;
        const uint16_t* xmv = master_v + (int64_t)li * S * E;
        build_agent_cache(sh, S, M, off + (int64_t)i * M, tok_block,
                          k_canon + (int64_t)l * S * E, v_canon + (int64_t)l * S * E,
                          sel + (int64_t)i * k, k,
                          k_fresh_sel + (((int64_t)i * nl + li) * k) * E,
                          v_fresh_sel + (((int64_t)i * nl + li) * k) * E, xik, xiv, c, s);
        for (int b = 0; b < nb; ++b) {
          int t0 = b * B, t1 = (b + 1) * B < S ? (b + 1) * B : S;
          size_t n = sizeof(uint16_t) * (size_t)(t1 - t0) * E;
          int differs = memcmp(xik + (int64_t)t0 * E, xmk + (int64_t)t0 * E, n) != 0 ||
                        memcmp(xiv + (int64_t)t0 * E, xmv + (int64_t)t0 * E, n) != 0;
          if (!differs) continue;
          if (write) {
            block_idx[nnz] = b;
            uint16_t* dk = val_k + nnz * B * E;
            uint16_t* dv = val_v + nnz * B * E;
            memset(dk, 0, sizeof(uint16_t) * B * E);
            memset(dv, 0, sizeof(uint16_t) * B * E);
            memcpy(dk, xik + (int64_t)t0 * E, n);
            memcpy(dv, xiv + (int64_t)t0 * E, n);
          }
          ++nnz;
        }
      }
    }
    if (write) rowptr[(int64_t)N * nl] = nnz;
  }
  *nnz_out = nnz;
  free(off); free(start); free(tok_block); free(c); free(s);
  free(xik); free(xiv);
  return status;
}

/* ------------------------------------------------------------------ stage 4 */
/* Fused diff restore: [R] Summary Method (3): on read-back, merge each diff into the
 * Master's data on its way and apply RoPE recovery, without building a dense Mirror;
 * §2a "Fused restore: Master chunk + diff -> paged KV"; §3d: recovery happens in the
 * transfer path and the result is written through the paged-KV slot map.
 * Each token's source is the agent's diff block when the agent is a Mirror with a record
 * for that (layer, block), else the Master; K is turned to the agent's offset (frame 0)
 * or copied as stored (frame 1); V is copied. Positions outside the shared span are not
 * touched. */
int orc_fused_restore(const orc_shape* sh, const orc_round* rd, int master,
                      const uint16_t* master_k, const uint16_t* master_v,
                      const int64_t* rowptr, const int32_t* block_idx,
                      const uint16_t* val_k, const uint16_t* val_v, const int32_t* agents,
                      int n_list, int layer_begin, int layer_end, int frame,
                      orc_pool* pool) {
  int N = rd->n_agents, M = rd->n_blocks, B = sh->diff_block, H = sh->n_kv_heads;
  int D = sh->head_dim;
  int64_t E = (int64_t)H * D;
  int S = shared_len(rd);
  int nl = layer_end - layer_begin;
  int nb = (S + B - 1) / B;
  if (master < 0 || master >= N) return ORC_ERR_ARG;
  int32_t* off = malloc(sizeof(int32_t) * N * M);
  int64_t* start = malloc(sizeof(int64_t) * (M + 1));
  int32_t* tok_block = malloc(sizeof(int32_t) * (S + 1));
  int64_t* row_of_block = malloc(sizeof(int64_t) * (nb > 0 ? nb : 1));
  float* c = malloc(sizeof(float) * D);
  float* s = malloc(sizeof(float) * D);
  int status = orc_offsets(rd, off);
  canon_layout(rd, start, tok_block);
  for (int x = 0; x < n_list && status == ORC_OK; ++x) {
    int a = agents[x];
    if (a < 0 || a >= N) { status = ORC_ERR_ARG; break; }
    for (int li = 0; li < nl; ++li) {
      int l = layer_begin + li;
      for (int b = 0; b < nb; ++b) row_of_block[b] = -1;
      if (a != master) {
        int64_t r0 = rowptr[(int64_t)a * nl + li], r1 = rowptr[(int64_t)a * nl + li + 1];
        for (int64_t r = r0; r < r1; ++r) row_of_block[block_idx[r]] = r;
      }
      for (int j = 0; j < M; ++j) {
        int32_t o = off[(int64_t)a * M + j];
        orc_rope_table(o, D, sh->rope_theta, c, s);
        for (int u = 0; u < rd->block_len[j]; ++u) {
          int64_t t = start[j] + u;
          int64_t r = row_of_block[t / B];
          const uint16_t* sk = r >= 0 ? val_k + (r * B + t % B) * E
                                      : master_k + ((int64_t)li * S + t) * E;
          const uint16_t* sv = r >= 0 ? val_v + (r * B + t % B) * E
                                      : master_v + ((int64_t)li * S + t) * E;
          int err = ORC_OK;
          uint16_t* kd = pool_row(sh, pool, a, l, 0, (int64_t)o + u, &err);
          if (!kd) { status = err; continue; }
          uint16_t* vd = pool_row(sh, pool, a, l, 1, (int64_t)o + u, &err);
          if (frame == 0) orc_rotate_row(sk, kd, H, D, c, s, 0);
          else memcpy(kd, sk, sizeof(uint16_t) * E);
          memcpy(vd, sv, sizeof(uint16_t) * E);
        }
      }
    }
  }
  free(off); free(start); free(tok_block); free(row_of_block); free(c); free(s);
  return status;
}

/* ------------------------------------------------------------------ attention */
/* Decode attention read straight from the Master and the diffs. [B] §4.4 "Fused Diff
 * Restore": the diff is applied block by block on chip and attention runs right after, with
 * no materialised cache; [R] §8 (open questions: the restore fused inside the attention
 * tile) and §9 (a paired block-sparse KV diff kernel aligned with FlashAttention).
 * READING: agent a's context is its private history, positions [0, h_a), whose K/V are read
 * from the paged pool as stored, followed by the shared blocks at their offsets: the shared
 * token t of block j at local index u sits at position off_aj + u with K = R(off_aj) X_a(t)
 * and V = X_a(t), X_a being the agent's canonical-frame cache (the Master's rows with a's
 * records over them). One query per (agent, query head), in the agent frame; query head g
 * reads kv head g / (n_q_heads / H). out = sum_p softmax_p(scale * q.k_p) v_p and
 * lse = log sum_p exp(scale * q.k_p). Everything in float64, the rotation of K exactly from
 * the bf16 values. The store holds exactly the layers [layer_begin, layer_end).
 * from_pool != 0: the same attention with every position [0, h_a + S) read from the pages
 * as stored (a restored cache); the store is not read. */
int orc_attention(const orc_shape* sh, const orc_round* rd, int master,
                  const uint16_t* master_k, const uint16_t* master_v,
                  const int64_t* rowptr, const int32_t* block_idx,
                  const uint16_t* val_k, const uint16_t* val_v, const orc_pool* pool,
                  const int32_t* agents, int n_list, int layer_begin, int layer_end,
                  const uint16_t* q, int n_q_heads, double scale, int from_pool, double* out,
                  double* lse) {
  int N = rd->n_agents, M = rd->n_blocks, B = sh->diff_block, H = sh->n_kv_heads;
  int D = sh->head_dim, P = sh->page_size;
  int64_t E = (int64_t)H * D;
  int S = shared_len(rd);
  int nl = layer_end - layer_begin;
  int nb = (S + B - 1) / B;
  if (master < 0 || master >= N || n_q_heads < H || n_q_heads % H != 0 || nl < 0)
    return ORC_ERR_ARG;
  int G = n_q_heads / H;
  int hmax = 0;
  for (int i = 0; i < N; ++i) hmax = rd->hist_len[i] > hmax ? rd->hist_len[i] : hmax;
  int64_t cap = (int64_t)hmax + S;
  int32_t* off = malloc(sizeof(int32_t) * N * M);
  int64_t* start = malloc(sizeof(int64_t) * (M + 1));
  int32_t* tok_block = malloc(sizeof(int32_t) * (S + 1));
  int64_t* row_of_block = malloc(sizeof(int64_t) * (nb > 0 ? nb : 1));
  double* kx = malloc(sizeof(double) * (cap > 0 ? cap : 1) * E);   /* the context's K */
  double* vx = malloc(sizeof(double) * (cap > 0 ? cap : 1) * E);   /* and V */
  double* sc = malloc(sizeof(double) * (cap > 0 ? cap : 1));
  int status = orc_offsets(rd, off);
  canon_layout(rd, start, tok_block);
  for (int li = 0; li < nl && status == ORC_OK; ++li) {
    int l = layer_begin + li;
    for (int x = 0; x < n_list && status == ORC_OK; ++x) {
      int a = agents[x];
      if (a < 0 || a >= N) { status = ORC_ERR_ARG; break; }
      int64_t n = (int64_t)rd->hist_len[a] + S;
      int64_t h = from_pool ? n : rd->hist_len[a];   /* positions read from the pages */
      /* the private history, as the pool holds it */
      for (int64_t p = 0; p < h && status == ORC_OK; ++p) {
        int64_t lp = p / P;
        int32_t page = lp < pool->max_lp ? pool->block_table[(int64_t)a * pool->max_lp + lp] : -1;
        if (page < 0 || page >= pool->num_pages) { status = ORC_ERR_UNMAPPED; break; }
        for (int kv = 0; kv < 2; ++kv) {
          const uint16_t* src = pool->base +
              ((((int64_t)l * 2 + kv) * pool->num_pages + page) * P + p % P) * E;
          double* dst = (kv == 0 ? kx : vx) + p * E;
          for (int64_t e = 0; e < E; ++e) dst[e] = (double)orc_bf16_to_f32(src[e]);
        }
      }
      /* the shared blocks: the agent's canonical cache, K turned to the agent's offsets */
      for (int b = 0; b < nb; ++b) row_of_block[b] = -1;
      if (a != master && !from_pool) {
        int64_t r0 = rowptr[(int64_t)a * nl + li], r1 = rowptr[(int64_t)a * nl + li + 1];
        for (int64_t r = r0; r < r1; ++r) row_of_block[block_idx[r]] = r;
      }
      for (int64_t t = 0; t < S && !from_pool; ++t) {
        int j = tok_block[t];
        int64_t r = row_of_block[t / B];
        const uint16_t* sk = r >= 0 ? val_k + (r * B + t % B) * E : master_k + ((int64_t)li * S + t) * E;
        const uint16_t* sv = r >= 0 ? val_v + (r * B + t % B) * E : master_v + ((int64_t)li * S + t) * E;
        orc_rotate_row_f64(sk, kx + (h + t) * E, H, D, off[(int64_t)a * M + j], sh->rope_theta, 0);
        for (int64_t e = 0; e < E; ++e) vx[(h + t) * E + e] = (double)orc_bf16_to_f32(sv[e]);
      }
      /* softmax attention of every query head over the n context positions */
      for (int g = 0; g < n_q_heads; ++g) {
        int hk = g / G;
        const uint16_t* qg = q + (((int64_t)li * n_list + x) * n_q_heads + g) * D;
        double* og = out + (((int64_t)li * n_list + x) * n_q_heads + g) * D;
        double mx = -INFINITY;
        for (int64_t p = 0; p < n; ++p) {
          double d = 0.0;
          for (int e = 0; e < D; ++e)
            d += (double)orc_bf16_to_f32(qg[e]) * kx[p * E + (int64_t)hk * D + e];
          sc[p] = scale * d;
          if (sc[p] > mx) mx = sc[p];
        }
        double sum = 0.0;
        for (int64_t p = 0; p < n; ++p) sum += exp(sc[p] - mx);
        for (int e = 0; e < D; ++e) {
          double acc = 0.0;
          for (int64_t p = 0; p < n; ++p) acc += exp(sc[p] - mx) * vx[p * E + (int64_t)hk * D + e];
          og[e] = n > 0 ? acc / sum : 0.0;
        }
        if (lse) lse[((int64_t)li * n_list + x) * n_q_heads + g] = n > 0 ? mx + log(sum) : -INFINITY;
      }
    }
  }
  free(off); free(start); free(tok_block); free(row_of_block); free(kx); free(vx); free(sc);
  return status;
}

/* ------------------------------------------------------------------ compression */
/* [R] §7a: compression ratio = dense KV size / (Master + diffs) size. Dense size of one
 * agent: L*S*E bf16 for K and again for V. A diff block costs its K and V values
 * (B*E*2 bytes each) plus its 4-byte index; the row pointers cost 8 bytes each.
 * READING: the round ratio compares N dense copies with one Master plus all diffs and
 * the row pointers; the per-Mirror ratio (the 11.2x / 17.5x of the "Storage Compression"
 * table) compares one dense copy with one Mirror's diff blocks. */
double orc_round_ratio(int n_agents, int n_layers, int n_shared, int elems, int diff_block,
                       int64_t nnz) {
  double dense = (double)n_layers * n_shared * elems * 2.0 * 2.0;
  double diff = (double)nnz * ((double)diff_block * elems * 4.0 + 4.0);
  double ptrs = 8.0 * ((double)n_agents * n_layers + 1.0);
  return (double)n_agents * dense / (dense + diff + ptrs);
}

double orc_mirror_ratio(int n_layers, int n_shared, int elems, int diff_block,
                        int64_t nnz_mirror) {
  double dense = (double)n_layers * n_shared * elems * 2.0 * 2.0;
  double diff = (double)nnz_mirror * ((double)diff_block * elems * 4.0 + 4.0);
  return dense / diff;
}
