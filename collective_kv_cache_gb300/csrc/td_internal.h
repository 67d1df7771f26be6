// td_internal.h - types shared by the host layer (td_host.cpp) and the kernels (*.cu).
#pragma once

#include <cuda.h>            // CUtensorMap: the attention kernels' tensor maps
#include <cuda_runtime.h>

#include <cstdint>

#include "td.h"

#ifdef __CUDACC__
#define TD_HD __host__ __device__
#else
#define TD_HD
#endif

namespace td {

constexpr int kTile = 16;          // canonical tokens per tile of the tile kernels
constexpr int kDiffBlock = 16;     // default tokens per diff block (canonical axis)
constexpr int kMaxDiffBlock = 32;  // diff blocks of 16 or 32 tokens (a 32-bit token mask)
constexpr int kMaxListAgents = 256; // agents per restore launch (passed by value)

TD_HD inline uint32_t err_bit(td_status s) { return 1u << static_cast<uint32_t>(s); }

// Token geometry of one model shape.
struct Geom {
  int H, D, E;   // heads, head_dim, elements per token row
  int half;      // D / 2
  int vpt;       // pair-vectors per token = E / 16 (8 frequencies of one head each)
};

// The current round's device tables (owned by the context).
struct RoundDev {
  int N, M, S;
  int B;                     // tokens per diff block (16 or 32, a multiple of kTile)
  int nb;                    // diff blocks, ceil(S / B)
  int nt;                    // tiles, ceil(S / kTile)
  const int32_t* off;        // [N*M] block start in each agent's prompt
  const float* cos_t;        // [N*M][D/2] cos of off * theta^(-2f/D), rounded to float
  const float* sin_t;        // [N*M][D/2]
  const int32_t* tok_block;  // [S] block of each canonical token
  const int32_t* blk_start;  // [M] canonical start of each block
  const int32_t* pos;        // [N][S] prompt position of each shared token, or nullptr
};

struct PoolDev {
  uint16_t* base;            // [L][2][num_pages][P][E]
  int64_t num_pages;
  const int32_t* bt;         // [N][max_lp]
  int max_lp;
  int P;
  int p_shift;               // log2(P) when P is a power of two, else -1
};

struct AgentList {
  int n;
  int32_t a[kMaxListAgents];
};

// Per-launch view of a diff store (offsets already relative to its first layer).
struct StoreDev {
  uint16_t* master_k;
  uint16_t* master_v;
  int64_t* rowptr;
  int32_t* block_idx;
  uint16_t* val_k;
  uint16_t* val_v;
  int32_t* slot;
  int64_t capacity;
  int nl;                    // layers held by the store
};

// Encode scratch (owned by the context).
struct EncodeScratch {
  uint32_t* selbits;         // [N][nb] selected tokens of agent i in diff block b (16 bits)
  int32_t* firstrank;        // [N][nb] rank in sel_i of the block's first selected token
  uint32_t* mask;            // [N][nbw] blocks holding a selected token of agent i
  uint32_t* cand;            // [N][nbw] mask_i | mask_m for i != m, 0 for the master
  int32_t* word_prefix;      // [N][nbw] candidates of agent i in words before w; then [N]
  int64_t* agent_prefix;     // [N+1] candidates per layer of agents before i
  uint32_t* flag;            // [N][nl][nb] candidate block differs from the master's
  int32_t* row_count;        // [N][nl] records per row; directly after flag (one memset)
  int32_t* words;            // [4]: unused, checked master, over capacity, prep counter
  int nbw;
};

// Threads per CTA of the tile kernels and items per thread (1 or 2).
int tile_threads(const Geom& g);
int tile_items(const Geom& g);

cudaError_t launch_rerotate(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                            const uint16_t* kc, const uint16_t* vc, int layer_begin, int nl,
                            uint32_t* err, cudaStream_t st);

// pos[i*S + t] = off[i*M + j(t)] + t - blk_start[j(t)] for the round's tables.
cudaError_t launch_positions(const RoundDev& rd, int32_t* pos, cudaStream_t st);

cudaError_t launch_deviation(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                             int check_layer, const uint16_t* k_fresh, float* dev,
                             uint32_t* err, cudaStream_t st);

cudaError_t launch_select(const float* dev, int N, int S, int k, int32_t* sel,
                          cudaStream_t st);

// Deviations, then the per-agent top-k (two launches). hist: [N][4096] first-digit counts,
// zero between calls (the top-k leaves them zero).
constexpr int kSelHistBins = 4096;
cudaError_t launch_check_select(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                int check_layer, const uint16_t* k_fresh, float* dev, int k,
                                int32_t* sel, uint32_t* hist, uint32_t* err, cudaStream_t st);

// gmask: [N][nbw] scratch; done: a counter that is zero between calls.
cudaError_t launch_pick_master(const int32_t* sel, int N, int S, int B, int k, int64_t* cost,
                               int32_t* master, uint32_t* gmask, int* done, uint32_t* err,
                               cudaStream_t st);

// Variant readings (k_variants.cu).
cudaError_t launch_min_dev_master(const int32_t* sel, const float* dev, int N, int S, int k,
                                  double* score, int32_t* master, uint32_t* err,
                                  cudaStream_t st);
cudaError_t launch_check_select_group(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                      int check_layer, const uint16_t* k_fresh, float* dev,
                                      float* gdev, int k, int32_t* sel, uint32_t* err,
                                      cudaStream_t st);

cudaError_t launch_encode(const Geom& g, const RoundDev& rd, const int32_t* master,
                          const uint16_t* kc, const uint16_t* vc, const int32_t* sel, int k,
                          const uint16_t* kf, const uint16_t* vf, int nl,
                          const StoreDev& store, const EncodeScratch& sc, uint32_t* err,
                          int64_t* bound_dev, cudaStream_t st);

cudaError_t launch_restore(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                           const StoreDev& store, const AgentList& agents, int layer_begin,
                           int store_layer0, int nl, int frame, uint32_t* err,
                           cudaStream_t st);

// Decode attention from the Master and the diffs (k_attention.cu).
constexpr int kAttnChunk = 512;    // context positions per work unit (one warp)
constexpr int kAttnTailChunk = 128; // ... in the units of the last layers (the grid's end)
constexpr int kAttnStage = 16;     // positions per pipeline stage
constexpr int kAttnDepth = 2;      // stages in flight per unit
constexpr int kAttnGMax = 8;       // query heads per kv head

// The units of a launch: layers [0, split) in units of kAttnChunk positions, then layers
// [split, nl) in units of kAttnTailChunk, so that the grid ends with short units and the
// SMs run full until close to the end.
struct AttnList {
  int n;                               // agents of this launch
  int split;                           // first layer (within the launch) of short units
  int32_t a[kMaxListAgents];           // their ids
  int32_t hist[kMaxListAgents];        // their history lengths
  int32_t base[kMaxListAgents + 1];    // exclusive prefix of their units (per layer, head)
  int32_t base2[kMaxListAgents + 1];   // the same in short units
};

struct AttnArgs {
  Geom g;
  RoundDev rd;
  PoolDev pool;
  StoreDev store;            // unused when every position comes from the pages
  const uint16_t* q;         // [nl][n_list][nq][D] bf16
  float* out;                // [nl][n_list][nq][D]
  float* lse;                // [nl][n_list][nq] or nullptr
  float* part_o;             // [units][G][D]
  float* part_ml;            // [units][G][2]: max, sum (base 2)
  int n_list, x0;            // the whole list's length; this launch's first entry
  int nq, G;                 // query heads, query heads per kv head
  int nl, layer_begin, sl0;  // layers; store layer of layer_begin
  float scale_log2;          // softmax scale * log2(e)
  uint32_t tx_pad;           // extra bytes every stage expects (fault injection; 0 normally)
  uint32_t* err;
};

// 2-D tensor maps ([rows][E] bf16, boxes of 16 rows x 64 columns, 128-byte swizzle) of the
// places the attention kernels stage rows from.
struct AttnMaps {
  CUtensorMap pool;          // rows = [L][2][num_pages][P]
  CUtensorMap master_k;      // rows = [nl][S]
  CUtensorMap master_v;
  CUtensorMap val_k;         // rows = [capacity][B]
  CUtensorMap val_v;
};

cudaError_t launch_attention(const AttnArgs& a, const AttnList& list, const AttnMaps& maps,
                             bool from_pool, cudaStream_t st);

cudaError_t launch_materialise(const Geom& g, const RoundDev& rd, const StoreDev& store,
                               int agent, int sl0, int nl, uint16_t* dk, uint16_t* dv,
                               uint32_t* err, cudaStream_t st);

}  // namespace td
