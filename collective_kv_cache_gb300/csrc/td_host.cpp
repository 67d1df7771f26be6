// td_host.cpp - the C ABI (include/td.h): argument validation, the context and its
// scratch, the round's offset and RoPE tables, and the kernel launches.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "td.h"
#include "td_internal.h"

using namespace td;

struct td_ctx {
  td_shape shape;
  Geom g;
  int max_agents, max_blocks, max_shared, max_nb, nbw_max;
  int device;

  // round tables (device) and their pinned staging
  int32_t* d_off = nullptr;
  float* d_cos = nullptr;
  float* d_sin = nullptr;
  int32_t* d_tok_block = nullptr;
  int32_t* d_blk_start = nullptr;
  unsigned char* h_stage = nullptr;
  size_t stage_bytes = 0;
  cudaEvent_t stage_done = nullptr;
  bool stage_pending = false;

  // Streams that have read the round tables since their last upload, each with an event
  // recorded after its latest launch. A round change makes the uploading stream wait on
  // all of them; a stream's first call after an upload waits on tables_ready.
  struct StreamUse {
    cudaStream_t stream;
    cudaEvent_t last_use;
    bool ordered;      // ordered after the current tables' upload
  };
  std::vector<StreamUse> users;
  cudaEvent_t tables_ready = nullptr;
  cudaStream_t tables_stream = nullptr;
  bool tables_recorded = false;

  // cached round (host copy) and its device view
  bool have_round = false;
  int N = 0, M = 0, S = 0;
  std::vector<int32_t> c_len, c_hist, c_perm;

  // scratch
  float* d_dev = nullptr;           // [max_agents * max_shared]
  int32_t* d_pos = nullptr;         // [max_agents * max_shared] prompt position of each token
  uint32_t* d_sel_hist = nullptr;   // [max_agents * kSelHistBins] selection histograms (zero)
  float* d_gdev = nullptr;          // [max_shared] group deviation (variant)
  double* d_score = nullptr;        // [max_agents] deviation totals (variant)
  uint32_t* d_selbits = nullptr;    // [max_agents * max_nb]
  int32_t* d_firstrank = nullptr;   // [max_agents * max_nb]
  uint32_t* d_mask = nullptr;       // [max_agents * nbw_max]
  uint32_t* d_cand = nullptr;       // [max_agents * nbw_max]
  uint32_t* d_pm_mask = nullptr;    // [max_agents * nbw_max] masks of td_pick_master
  int32_t* d_wprefix = nullptr;     // [max_agents * nbw_max + max_agents]
  int64_t* d_aprefix = nullptr;     // [max_agents + 1]
  uint32_t* d_flag = nullptr;       // [max_agents * L * max_nb] flags + [max_agents * L] counts
  int sm_count = 0;                 // of the context's device
  int32_t* d_ints = nullptr;        // encode's words (unused, m_ok, over, prep_done), spare,
                                    // pick_master's counter, spare
  int64_t* d_bound = nullptr;
  uint32_t* d_err = nullptr;
  float* d_attn = nullptr;          // attention partials, grown on demand
  size_t attn_cap = 0;              // its size in floats
  uint32_t attn_tx_pad = 0;         // fault injection: bytes the attention never receives
  // pinned host words for results
  int64_t* h_words = nullptr;       // [4]
};

namespace {

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

void free_ctx(td_ctx* c) {
  if (!c) return;
  cudaFree(c->d_off);
  cudaFree(c->d_cos);
  cudaFree(c->d_sin);
  cudaFree(c->d_tok_block);
  cudaFree(c->d_blk_start);
  cudaFree(c->d_dev);
  cudaFree(c->d_pos);
  cudaFree(c->d_sel_hist);
  cudaFree(c->d_gdev);
  cudaFree(c->d_score);
  cudaFree(c->d_selbits);
  cudaFree(c->d_firstrank);
  cudaFree(c->d_mask);
  cudaFree(c->d_cand);
  cudaFree(c->d_pm_mask);
  cudaFree(c->d_wprefix);
  cudaFree(c->d_aprefix);
  cudaFree(c->d_flag);
  cudaFree(c->d_ints);
  cudaFree(c->d_bound);
  cudaFree(c->d_err);
  cudaFree(c->d_attn);
  if (c->h_stage) cudaFreeHost(c->h_stage);
  if (c->h_words) cudaFreeHost(c->h_words);
  if (c->stage_done) cudaEventDestroy(c->stage_done);
  if (c->tables_ready) cudaEventDestroy(c->tables_ready);
  for (auto& u : c->users) cudaEventDestroy(u.last_use);
  delete c;
}

bool same_device(const td_ctx* c) {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess && d == c->device;
}

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

td_ctx::StreamUse* find_use(td_ctx* c, cudaStream_t st) {
  for (auto& u : c->users)
    if (u.stream == st) return &u;
  return nullptr;
}

constexpr size_t kMaxTrackedStreams = 64;

// The entry of `st` in the users list, created when missing (when the list is full, every
// tracked stream is first drained on the host and the list starts over).
td_ctx::StreamUse* use_of(td_ctx* c, cudaStream_t st) {
  if (td_ctx::StreamUse* u = find_use(c, st)) return u;
  if (c->users.size() >= kMaxTrackedStreams) {
    for (auto& u : c->users) {
      if (cudaEventSynchronize(u.last_use) != cudaSuccess) return nullptr;
      cudaEventDestroy(u.last_use);
    }
    c->users.clear();
  }
  td_ctx::StreamUse u{st, nullptr, false};
  if (cudaEventCreateWithFlags(&u.last_use, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  // a fresh event counts as complete: waiting on it before its first record is a no-op
  c->users.push_back(u);
  return &c->users.back();
}

// Orders `st` after the upload of the current tables (once per stream and upload).
td_status order_after_tables(td_ctx* c, cudaStream_t st) {
  td_ctx::StreamUse* u = use_of(c, st);
  if (!u) return TD_ERR_CUDA;
  if (u->ordered) return TD_OK;
  if (c->tables_recorded && st != c->tables_stream &&
      cudaStreamWaitEvent(st, c->tables_ready, 0) != cudaSuccess)
    return TD_ERR_CUDA;
  u->ordered = true;
  return TD_OK;
}

// After a call's launches: its stream's reads of the tables end with this point.
td_status note_use(td_ctx* c, cudaStream_t st) {
  if (capturing(st)) return TD_OK;
  td_ctx::StreamUse* u = find_use(c, st);
  if (!u) return TD_OK;
  return cudaEventRecord(u->last_use, st) == cudaSuccess ? TD_OK : TD_ERR_CUDA;
}

// Validates the round and brings the device tables up to date with it. The tables are
// shared by every stream that uses the context: a stream is ordered after their upload
// before its first launch, and a new upload waits (on the device) for every launch that
// may still read the old tables. Inside a stream capture nothing is tracked and a change
// of round is refused: the tables must already hold the round, uploaded and finished.
td_status prepare_round(td_ctx* c, const td_round* r, cudaStream_t st) {
  if (!r || !r->block_len || !r->hist_len || !r->perm) return TD_ERR_INVALID_ARG;
  const int N = r->n_agents, M = r->n_blocks;
  if (N < 1 || N > c->max_agents || M < 1 || M > c->max_blocks) return TD_ERR_INVALID_ARG;
  int64_t S = 0;
  for (int j = 0; j < M; ++j) {
    if (r->block_len[j] < 1) return TD_ERR_INVALID_ARG;
    S += r->block_len[j];
  }
  if (S > c->max_shared) return TD_ERR_INVALID_ARG;
  for (int i = 0; i < N; ++i) {
    if (r->hist_len[i] < 0 || static_cast<int64_t>(r->hist_len[i]) + S > INT32_MAX / 2)
      return TD_ERR_INVALID_ARG;
    std::vector<char> seen(M, 0);
    for (int q = 0; q < M; ++q) {
      const int j = r->perm[static_cast<int64_t>(i) * M + q];
      if (j < 0 || j >= M || seen[j]) return TD_ERR_INVALID_ARG;
      seen[j] = 1;
    }
  }
  const bool cap = capturing(st);
  if (c->have_round && c->N == N && c->M == M &&
      std::memcmp(c->c_len.data(), r->block_len, sizeof(int32_t) * M) == 0 &&
      std::memcmp(c->c_hist.data(), r->hist_len, sizeof(int32_t) * N) == 0 &&
      std::memcmp(c->c_perm.data(), r->perm, sizeof(int32_t) * N * M) == 0)
    return cap ? TD_OK : order_after_tables(c, st);
  if (cap) return TD_ERR_INVALID_ARG;

  // every launch that may still read the old tables finishes before they change
  for (auto& u : c->users)
    if (u.stream != st && cudaStreamWaitEvent(st, u.last_use, 0) != cudaSuccess)
      return TD_ERR_CUDA;

  // the previous upload must have left the staging buffer before it is rewritten
  if (c->stage_pending) {
    if (cudaEventSynchronize(c->stage_done) != cudaSuccess) return TD_ERR_CUDA;
    c->stage_pending = false;
  }
  const int half = c->g.half;
  const size_t n_off = static_cast<size_t>(N) * M;
  unsigned char* p = c->h_stage;
  int32_t* off = reinterpret_cast<int32_t*>(p);
  float* cs = reinterpret_cast<float*>(off + n_off);
  float* sn = cs + n_off * half;
  int32_t* tokb = reinterpret_cast<int32_t*>(sn + n_off * half);
  int32_t* bst = tokb + S;
  // offsets: history, then the blocks in the agent's order
  for (int i = 0; i < N; ++i) {
    int64_t pos = r->hist_len[i];
    for (int q = 0; q < M; ++q) {
      const int j = r->perm[static_cast<int64_t>(i) * M + q];
      off[static_cast<int64_t>(i) * M + j] = static_cast<int32_t>(pos);
      pos += r->block_len[j];
    }
  }
  // RoPE tables: angle = off * theta^(-2f/D) in float64, cos/sin rounded once to float
  std::vector<double> inv_freq(half);
  for (int f = 0; f < half; ++f)
    inv_freq[f] = std::pow(c->shape.rope_theta,
                           -static_cast<double>(2 * f) / static_cast<double>(c->g.D));
  for (size_t ab = 0; ab < n_off; ++ab) {
    const double a = static_cast<double>(off[ab]);
    for (int f = 0; f < half; ++f) {
      const double ang = a * inv_freq[f];
      cs[ab * half + f] = static_cast<float>(std::cos(ang));
      sn[ab * half + f] = static_cast<float>(std::sin(ang));
    }
  }
  int64_t s0 = 0;
  for (int j = 0; j < M; ++j) {
    bst[j] = static_cast<int32_t>(s0);
    for (int u = 0; u < r->block_len[j]; ++u) tokb[s0 + u] = j;
    s0 += r->block_len[j];
  }
  cudaError_t e;
  if ((e = cudaMemcpyAsync(c->d_off, off, n_off * 4, cudaMemcpyHostToDevice, st)) ||
      (e = cudaMemcpyAsync(c->d_cos, cs, n_off * half * 4, cudaMemcpyHostToDevice, st)) ||
      (e = cudaMemcpyAsync(c->d_sin, sn, n_off * half * 4, cudaMemcpyHostToDevice, st)) ||
      (e = cudaMemcpyAsync(c->d_tok_block, tokb, S * 4, cudaMemcpyHostToDevice, st)) ||
      (e = cudaMemcpyAsync(c->d_blk_start, bst, M * 4, cudaMemcpyHostToDevice, st)) ||
      (e = cudaEventRecord(c->stage_done, st)))
    return TD_ERR_CUDA;
  {
    RoundDev rd{};
    rd.N = N;
    rd.M = M;
    rd.S = static_cast<int>(S);
    rd.off = c->d_off;
    rd.tok_block = c->d_tok_block;
    rd.blk_start = c->d_blk_start;
    if ((e = launch_positions(rd, c->d_pos, st)) || (e = cudaEventRecord(c->tables_ready, st)))
      return TD_ERR_CUDA;
  }
  c->tables_stream = st;
  c->tables_recorded = true;
  for (auto& u : c->users) u.ordered = false;
  if (order_after_tables(c, st) != TD_OK) return TD_ERR_CUDA;
  c->stage_pending = true;
  c->have_round = true;
  c->N = N;
  c->M = M;
  c->S = static_cast<int>(S);
  c->c_len.assign(r->block_len, r->block_len + M);
  c->c_hist.assign(r->hist_len, r->hist_len + N);
  c->c_perm.assign(r->perm, r->perm + static_cast<size_t>(N) * M);
  return TD_OK;
}

RoundDev round_dev(const td_ctx* c) {
  RoundDev rd;
  rd.N = c->N;
  rd.M = c->M;
  rd.S = c->S;
  rd.B = c->shape.diff_block;
  rd.nb = (c->S + rd.B - 1) / rd.B;
  rd.nt = (c->S + kTile - 1) / kTile;
  rd.off = c->d_off;
  rd.cos_t = c->d_cos;
  rd.sin_t = c->d_sin;
  rd.tok_block = c->d_tok_block;
  rd.blk_start = c->d_blk_start;
  rd.pos = c->d_pos;
  return rd;
}

// The pool must map every shared position: hist + S - 1 fits the block table.
td_status pool_dev(const td_ctx* c, const td_round* r, const td_paged* p, PoolDev* out) {
  if (!p || !p->base || !p->block_table || p->num_pages < 1 || p->max_pages_per_agent < 1)
    return TD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(p->base) & 15u) != 0) return TD_ERR_INVALID_ARG;
  const int P = c->shape.page_size;
  for (int i = 0; i < r->n_agents; ++i) {
    const int64_t last = static_cast<int64_t>(r->hist_len[i]) + c->S - 1;
    if (last / P >= p->max_pages_per_agent) return TD_ERR_INVALID_ARG;
  }
  out->base = static_cast<uint16_t*>(p->base);
  out->num_pages = p->num_pages;
  out->bt = p->block_table;
  out->max_lp = p->max_pages_per_agent;
  out->P = P;
  out->p_shift = is_pow2(P) ? log2i(P) : -1;
  return TD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A [rows][E] bf16 array as a 2-D tensor map with 16 x 64 boxes and 128-byte swizzle.
bool row_map(CUtensorMap* m, const void* base, uint64_t rows, int E) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn || !base || rows == 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(E) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kAttnStage)};
  const cuuint32_t elem[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Decode attention of the listed agents: shared positions from the store (store != null)
// or every position from the pages (store == null, the restored cache).
td_status run_attention(td_ctx* c, const td_round* r, const td_diff_store* store,
                        const td_paged* pool, const int32_t* agents, int32_t n_list,
                        int32_t layer_begin, int32_t layer_end, const void* q,
                        int32_t n_q_heads, float scale, float* out, float* lse, void* stream) {
  if (!c || !same_device(c) || n_list < 0 || (n_list > 0 && (!agents || !q || !out)))
    return TD_ERR_INVALID_ARG;
  const int H = c->g.H, D = c->g.D;
  if ((D != 64 && D != 128) || n_q_heads < H || n_q_heads % H != 0 ||
      n_q_heads / H > kAttnGMax || !std::isfinite(scale))
    return TD_ERR_INVALID_ARG;
  if (layer_begin < 0 || layer_end > c->shape.n_layers || layer_begin >= layer_end)
    return TD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 3u) != 0) return TD_ERR_INVALID_ARG;
  if (store) {
    if (!store->master_k || !store->master_v || !store->slot || !aligned16(store->master_k) ||
        !aligned16(store->master_v) || (store->val_k && !aligned16(store->val_k)) ||
        (store->val_v && !aligned16(store->val_v)))
      return TD_ERR_INVALID_ARG;
    if (layer_begin < store->layer_begin || layer_end > store->layer_end ||
        store->layer_begin < 0 || store->layer_end > c->shape.n_layers)
      return TD_ERR_INVALID_ARG;
    // the rows are staged by the bulk-copy engine from device memory only
    const void* ptrs[] = {store->master_k, store->master_v, store->slot, store->val_k,
                          store->val_v};
    for (const void* p : ptrs) {
      if (!p) continue;
      cudaPointerAttributes at;
      if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return TD_ERR_INVALID_ARG;
      }
      if (at.type != cudaMemoryTypeDevice) return TD_ERR_INVALID_ARG;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  for (int x = 0; x < n_list; ++x)
    if (agents[x] < 0 || agents[x] >= c->N) return TD_ERR_INVALID_ARG;
  if (n_list == 0) return TD_OK;
  PoolDev pd;
  if ((s = pool_dev(c, r, pool, &pd)) != TD_OK) return s;
  AttnArgs a{};
  a.g = c->g;
  a.rd = round_dev(c);
  a.pool = pd;
  if (store) {
    a.store.master_k = static_cast<uint16_t*>(store->master_k);
    a.store.master_v = static_cast<uint16_t*>(store->master_v);
    a.store.rowptr = store->rowptr;
    a.store.block_idx = store->block_idx;
    a.store.val_k = static_cast<uint16_t*>(store->val_k);
    a.store.val_v = static_cast<uint16_t*>(store->val_v);
    a.store.slot = store->slot;
    a.store.capacity = store->capacity_blocks;
    a.store.nl = store->layer_end - store->layer_begin;
    a.sl0 = layer_begin - store->layer_begin;
  }
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.lse = lse;
  a.n_list = n_list;
  a.nq = n_q_heads;
  a.G = n_q_heads / H;
  a.nl = layer_end - layer_begin;
  a.layer_begin = layer_begin;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.tx_pad = c->attn_tx_pad;
  a.err = c->d_err;
  // an agent's units: its history, then its shared tokens, each in chunks of `ch`
  // positions (every position from the pages: the whole context in chunks)
  auto units_of = [&](int x, int ch) -> int64_t {
    const int64_t hl = r->hist_len[agents[x]];
    if (!store) return (hl + c->S + ch - 1) / ch;
    return (hl + ch - 1) / ch + (c->S + ch - 1) / ch;
  };
  // The grid ends with the last layers in short units, about half a wave of the machine
  // (13 warps an SM, each on kAttnChunk positions), so that the last units to start are
  // short. Only where a layer is less than half a wave and the grid is more than one wave:
  // in larger layers the final wave is a small part of the call, and a whole layer in short
  // units would cost more partials than its tail saves; a grid of one wave or less has no
  // last wave to shorten, only more partials to combine.
  const int nl = layer_end - layer_begin;
  int n_short = 0;
  {
    int64_t per_layer = 0;   // context positions of one layer of the first agent list
    int64_t long_units = 0;  // its units of kAttnChunk positions
    for (int x = 0; x < n_list && x < kMaxListAgents; ++x) {
      per_layer += static_cast<int64_t>(r->hist_len[agents[x]]) + c->S;
      long_units += units_of(x, kAttnChunk);
    }
    per_layer *= H;
    long_units *= static_cast<int64_t>(H) * nl;
    const int64_t wave = static_cast<int64_t>(c->sm_count) * 13;
    const int64_t half_wave = wave * kAttnChunk / 2;
    if (per_layer > 0 && per_layer <= half_wave && long_units > wave) {
      const int64_t t = (half_wave + per_layer - 1) / per_layer;
      n_short = static_cast<int>(t > nl - 1 ? nl - 1 : t);
    }
  }
  const int split = nl - n_short;
  // partials of the largest agent list; grown once, after the work that used them
  int64_t most = 0;
  for (int x0 = 0; x0 < n_list; x0 += kMaxListAgents) {
    int64_t sum = 0;
    for (int x = x0; x < n_list && x < x0 + kMaxListAgents; ++x)
      sum += units_of(x, kAttnChunk) * split + units_of(x, kAttnTailChunk) * n_short;
    most = sum > most ? sum : most;
  }
  AttnMaps maps;
  const uint64_t pool_rows = static_cast<uint64_t>(c->shape.n_layers) * 2 *
                             static_cast<uint64_t>(pd.num_pages) * pd.P;
  if (!row_map(&maps.pool, pd.base, pool_rows, c->g.E)) return TD_ERR_CUDA;
  if (store) {
    const uint64_t mrows = static_cast<uint64_t>(a.store.nl) * c->S;
    const uint64_t vrows = static_cast<uint64_t>(store->capacity_blocks) * c->shape.diff_block;
    if (!row_map(&maps.master_k, store->master_k, mrows, c->g.E) ||
        !row_map(&maps.master_v, store->master_v, mrows, c->g.E))
      return TD_ERR_CUDA;
    const bool recs = vrows > 0 && store->val_k && store->val_v;
    if (!row_map(&maps.val_k, recs ? store->val_k : store->master_k, recs ? vrows : mrows,
                 c->g.E) ||
        !row_map(&maps.val_v, recs ? store->val_v : store->master_v, recs ? vrows : mrows,
                 c->g.E))
      return TD_ERR_CUDA;
  } else {
    maps.master_k = maps.master_v = maps.val_k = maps.val_v = maps.pool;
  }
  const size_t need = static_cast<size_t>(most) * H * kAttnGMax * (D + 2);
  if (need > c->attn_cap) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return TD_ERR_CUDA;
    cudaFree(c->d_attn);
    c->d_attn = nullptr;
    c->attn_cap = 0;
    if (cudaMalloc(&c->d_attn, need * sizeof(float)) != cudaSuccess) return TD_ERR_CUDA;
    c->attn_cap = need;
  }
  for (int x0 = 0; x0 < n_list; x0 += kMaxListAgents) {
    AttnList L;
    L.n = n_list - x0 < kMaxListAgents ? n_list - x0 : kMaxListAgents;
    L.split = split;
    L.base[0] = L.base2[0] = 0;
    for (int x = 0; x < L.n; ++x) {
      L.a[x] = agents[x0 + x];
      L.hist[x] = r->hist_len[agents[x0 + x]];
      const int64_t nb = L.base[x] + units_of(x0 + x, kAttnChunk);
      const int64_t nb2 = L.base2[x] + units_of(x0 + x, kAttnTailChunk);
      if (nb > INT32_MAX || nb2 > INT32_MAX) return TD_ERR_INVALID_ARG;
      L.base[x + 1] = static_cast<int32_t>(nb);
      L.base2[x + 1] = static_cast<int32_t>(nb2);
    }
    const int64_t units = static_cast<int64_t>(L.base[L.n]) * split * H +
                          static_cast<int64_t>(L.base2[L.n]) * n_short * H;
    if (units > INT32_MAX) return TD_ERR_INVALID_ARG;
    a.x0 = x0;
    a.part_o = c->d_attn;
    a.part_ml = c->d_attn + static_cast<size_t>(units) * kAttnGMax * D;
    if (launch_attention(a, L, maps, store == nullptr, st) != cudaSuccess) return TD_ERR_CUDA;
  }
  return note_use(c, st);
}

}  // namespace

extern "C" {

const char* td_status_string(td_status s) {
  switch (s) {
    case TD_OK: return "ok";
    case TD_ERR_INVALID_ARG: return "invalid argument";
    case TD_ERR_CUDA: return "CUDA error";
    case TD_ERR_CAPACITY: return "diff store capacity exceeded";
    case TD_ERR_UNMAPPED_PAGE: return "unmapped or out-of-range page";
    case TD_ERR_NONFINITE: return "non-finite key deviation";
    case TD_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case TD_ERR_SCRATCH_LIMIT: return "round exceeds the fixed scratch of td_check_select_noalloc";
  }
  return "unknown status";
}

td_status td_ctx_create(const td_shape* shape, int32_t max_agents, int32_t max_blocks,
                        int32_t max_shared, td_ctx** out) {
  if (!shape || !out) return TD_ERR_INVALID_ARG;
  *out = nullptr;
  const td_shape& s = *shape;
  if (s.n_layers < 1 || s.n_kv_heads < 1 || s.head_dim < 16 || s.head_dim % 16 != 0 ||
      s.page_size < 1 || (s.diff_block != 16 && s.diff_block != kMaxDiffBlock) || !(s.rope_theta > 1.0) ||
      !std::isfinite(s.rope_theta))
    return TD_ERR_INVALID_ARG;
  const int64_t E = static_cast<int64_t>(s.n_kv_heads) * s.head_dim;
  if (E > 2048) return TD_ERR_INVALID_ARG;  // a tile holds 16 rows of at most 2048 elements
  if (max_agents < 1 || max_blocks < 1 || max_shared < 1 || max_agents > 4096 ||
      max_shared > (1 << 22))
    return TD_ERR_INVALID_ARG;
  const int max_nb = (max_shared + kDiffBlock - 1) / kDiffBlock;
  const int nbw = (max_nb + 31) / 32;
  // one-CTA kernels keep per-agent masks and per-row counts in shared memory
  if (static_cast<int64_t>(max_agents) * nbw * 4 + 8 * max_agents > 160 * 1024) return TD_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_agents) * s.n_layers * 8 > 160 * 1024) return TD_ERR_INVALID_ARG;

  td_ctx* c = new (std::nothrow) td_ctx;
  if (!c) return TD_ERR_CUDA;
  c->shape = s;
  c->g.H = s.n_kv_heads;
  c->g.D = s.head_dim;
  c->g.E = static_cast<int>(E);
  c->g.half = s.head_dim / 2;
  c->g.vpt = static_cast<int>(E / 16);
  c->max_agents = max_agents;
  c->max_blocks = max_blocks;
  c->max_shared = max_shared;
  c->max_nb = max_nb;
  c->nbw_max = nbw;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device) !=
          cudaSuccess) {
    delete c;
    return TD_ERR_CUDA;
  }
  const size_t NM = static_cast<size_t>(max_agents) * max_blocks;
  const size_t half = c->g.half;
  const size_t NS = static_cast<size_t>(max_agents) * max_shared;
  c->stage_bytes = NM * 4 + 2 * NM * half * 4 + static_cast<size_t>(max_shared) * 4 + max_blocks * 4 + 64;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t x) { if (e == cudaSuccess) e = x; };
  chk(cudaMalloc(&c->d_off, NM * 4));
  chk(cudaMalloc(&c->d_cos, NM * half * 4));
  chk(cudaMalloc(&c->d_sin, NM * half * 4));
  chk(cudaMalloc(&c->d_tok_block, static_cast<size_t>(max_shared) * 4));
  chk(cudaMalloc(&c->d_blk_start, static_cast<size_t>(max_blocks) * 4));
  chk(cudaMalloc(&c->d_dev, NS * 4));
  chk(cudaMalloc(&c->d_pos, NS * 4));
  chk(cudaMalloc(&c->d_sel_hist, static_cast<size_t>(max_agents) * kSelHistBins * 4));
  chk(cudaMalloc(&c->d_gdev, static_cast<size_t>(max_shared) * 4));
  chk(cudaMalloc(&c->d_score, static_cast<size_t>(max_agents) * 8));
  chk(cudaMalloc(&c->d_selbits, static_cast<size_t>(max_agents) * max_nb * 4));
  chk(cudaMalloc(&c->d_firstrank, static_cast<size_t>(max_agents) * max_nb * 4));
  chk(cudaMalloc(&c->d_mask, static_cast<size_t>(max_agents) * nbw * 4));
  chk(cudaMalloc(&c->d_cand, static_cast<size_t>(max_agents) * nbw * 4));
  chk(cudaMalloc(&c->d_pm_mask, static_cast<size_t>(max_agents) * nbw * 4));
  chk(cudaMalloc(&c->d_wprefix, (static_cast<size_t>(max_agents) * nbw + max_agents) * 4));
  chk(cudaMalloc(&c->d_aprefix, (static_cast<size_t>(max_agents) + 1) * 8));
  chk(cudaMalloc(&c->d_flag, (static_cast<size_t>(max_agents) * s.n_layers * max_nb +
                              static_cast<size_t>(max_agents) * s.n_layers) * 4));
  chk(cudaMalloc(&c->d_ints, 8 * sizeof(int32_t)));
  chk(cudaMalloc(&c->d_bound, sizeof(int64_t)));
  chk(cudaMalloc(&c->d_err, sizeof(uint32_t)));
  chk(cudaMallocHost(&c->h_stage, c->stage_bytes));
  chk(cudaMallocHost(&c->h_words, 4 * sizeof(int64_t)));
  chk(cudaEventCreateWithFlags(&c->stage_done, cudaEventDisableTiming));
  chk(cudaEventCreateWithFlags(&c->tables_ready, cudaEventDisableTiming));
  if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d_ints, 0, 8 * sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaMemset(c->d_sel_hist, 0, static_cast<size_t>(max_agents) * kSelHistBins * 4);
  if (e != cudaSuccess) {
    free_ctx(c);
    return TD_ERR_CUDA;
  }
  *out = c;
  return TD_OK;
}

td_status td_ctx_destroy(td_ctx* ctx) {
  if (!ctx) return TD_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  free_ctx(ctx);
  return TD_OK;
}

td_status td_round_offsets(const td_round* r, int32_t* off_out) {
  if (!r || !off_out || !r->block_len || !r->hist_len || !r->perm || r->n_agents < 1 ||
      r->n_blocks < 1)
    return TD_ERR_INVALID_ARG;
  const int N = r->n_agents, M = r->n_blocks;
  for (int i = 0; i < N; ++i) {
    std::vector<char> seen(M, 0);
    int64_t pos = r->hist_len[i];
    if (pos < 0) return TD_ERR_INVALID_ARG;
    for (int q = 0; q < M; ++q) {
      const int j = r->perm[static_cast<int64_t>(i) * M + q];
      if (j < 0 || j >= M || seen[j] || r->block_len[j] < 1) return TD_ERR_INVALID_ARG;
      seen[j] = 1;
      if (pos > INT32_MAX) return TD_ERR_INVALID_ARG;
      off_out[static_cast<int64_t>(i) * M + j] = static_cast<int32_t>(pos);
      pos += r->block_len[j];
    }
  }
  return TD_OK;
}

td_status td_rerotate_batched(td_ctx* c, const td_round* r, const void* k_canon,
                              const void* v_canon, int32_t layer_begin, int32_t layer_end,
                              const td_paged* pool, void* stream) {
  if (!c || !same_device(c) || !k_canon || !aligned16(k_canon) ||
      (v_canon && !aligned16(v_canon)))
    return TD_ERR_INVALID_ARG;
  if (layer_begin < 0 || layer_end > c->shape.n_layers || layer_begin > layer_end)
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  PoolDev pd;
  if ((s = pool_dev(c, r, pool, &pd)) != TD_OK) return s;
  if (launch_rerotate(c->g, round_dev(c), pd, static_cast<const uint16_t*>(k_canon),
                      static_cast<const uint16_t*>(v_canon), layer_begin, layer_end - layer_begin,
                      c->d_err, st) != cudaSuccess)
    return TD_ERR_CUDA;
  return note_use(c, st);
}

td_status td_check_select(td_ctx* c, const td_round* r, int32_t check_layer,
                          const td_paged* pool, const void* k_fresh, int32_t recompute_pct,
                          int32_t* sel, float* dev_out, int32_t* k_out, void* stream) {
  if (!c || !same_device(c) || !k_fresh || !aligned16(k_fresh) || !k_out)
    return TD_ERR_INVALID_ARG;
  if (check_layer < 0 || check_layer >= c->shape.n_layers || recompute_pct < 0 ||
      recompute_pct > 100)
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  PoolDev pd;
  if ((s = pool_dev(c, r, pool, &pd)) != TD_OK) return s;
  const int k = static_cast<int>((static_cast<int64_t>(recompute_pct) * c->S + 99) / 100);
  if (k > 0 && !sel) return TD_ERR_INVALID_ARG;
  *k_out = k;
  float* dev = dev_out ? dev_out : c->d_dev;
  const RoundDev rd = round_dev(c);
  if (launch_check_select(c->g, rd, pd, check_layer, static_cast<const uint16_t*>(k_fresh), dev,
                          k, sel, c->d_sel_hist, c->d_err, st) != cudaSuccess)
    return TD_ERR_CUDA;
  return note_use(c, st);
}

td_status td_pick_master(td_ctx* c, const td_round* r, const int32_t* sel, int32_t k,
                         int64_t* cost_out, int32_t* master_dev, int32_t* master_host,
                         void* stream) {
  if (!c || !same_device(c) || !master_dev || k < 0 || (k > 0 && !sel))
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  if (k > c->S) return TD_ERR_INVALID_ARG;
  cudaError_t e = launch_pick_master(sel, c->N, c->S, c->shape.diff_block, k, cost_out, master_dev, c->d_pm_mask,
                                     c->d_ints + 5, c->d_err, st);
  if (e != cudaSuccess || note_use(c, st) != TD_OK) return TD_ERR_CUDA;
  if (master_host) {
    int32_t* h = reinterpret_cast<int32_t*>(c->h_words);
    if ((e = cudaMemcpyAsync(h, master_dev, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)
      return TD_ERR_CUDA;
    *master_host = *h;
  }
  return TD_OK;
}

td_status td_check_select_group(td_ctx* c, const td_round* r, int32_t check_layer,
                                const td_paged* pool, const void* k_fresh,
                                int32_t recompute_pct, int32_t* sel, float* dev_out,
                                float* group_dev_out, int32_t* k_out, void* stream) {
  if (!c || !same_device(c) || !k_fresh || !aligned16(k_fresh) || !k_out)
    return TD_ERR_INVALID_ARG;
  if (check_layer < 0 || check_layer >= c->shape.n_layers || recompute_pct < 0 ||
      recompute_pct > 100)
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  PoolDev pd;
  if ((s = pool_dev(c, r, pool, &pd)) != TD_OK) return s;
  const int k = static_cast<int>((static_cast<int64_t>(recompute_pct) * c->S + 99) / 100);
  if (k > 0 && !sel) return TD_ERR_INVALID_ARG;
  *k_out = k;
  if (launch_check_select_group(c->g, round_dev(c), pd, check_layer,
                                static_cast<const uint16_t*>(k_fresh),
                                dev_out ? dev_out : c->d_dev,
                                group_dev_out ? group_dev_out : c->d_gdev, k, sel, c->d_err,
                                st) != cudaSuccess)
    return TD_ERR_CUDA;
  return note_use(c, st);
}

td_status td_pick_master_min_deviation(td_ctx* c, const td_round* r, const int32_t* sel,
                                       int32_t k, const float* dev, double* score_out,
                                       int32_t* master_dev, int32_t* master_host,
                                       void* stream) {
  if (!c || !same_device(c) || !master_dev || !dev || k < 0 || (k > 0 && !sel))
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  if (k > c->S) return TD_ERR_INVALID_ARG;
  cudaError_t e = launch_min_dev_master(sel, dev, c->N, c->S, k,
                                        score_out ? score_out : c->d_score, master_dev,
                                        c->d_err, st);
  if (e != cudaSuccess || note_use(c, st) != TD_OK) return TD_ERR_CUDA;
  if (master_host) {
    int32_t* h = reinterpret_cast<int32_t*>(c->h_words);
    if (cudaMemcpyAsync(h, master_dev, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return TD_ERR_CUDA;
    *master_host = *h;
  }
  return TD_OK;
}

td_status td_diff_encode(td_ctx* c, const td_round* r, const int32_t* master,
                         const void* k_canon, const void* v_canon, const int32_t* sel,
                         int32_t k, const void* k_fresh_sel, const void* v_fresh_sel,
                         int32_t layer_begin, int32_t layer_end, td_diff_store* store,
                         int64_t* nnz_out, void* stream) {
  if (!c || !same_device(c) || !master || !k_canon || !v_canon || !store ||
      !aligned16(k_canon) || !aligned16(v_canon))
    return TD_ERR_INVALID_ARG;
  if (k < 0 || (k > 0 && (!sel || !k_fresh_sel || !v_fresh_sel || !aligned16(k_fresh_sel) ||
                          !aligned16(v_fresh_sel))))
    return TD_ERR_INVALID_ARG;
  if (layer_begin < 0 || layer_end > c->shape.n_layers || layer_begin >= layer_end)
    return TD_ERR_INVALID_ARG;
  if (!store->master_k || !store->master_v || !store->rowptr || !store->slot ||
      !aligned16(store->master_k) || !aligned16(store->master_v) || store->capacity_blocks < 0)
    return TD_ERR_INVALID_ARG;
  if (store->capacity_blocks > 0 &&
      (!store->block_idx || !store->val_k || !store->val_v || !aligned16(store->val_k) ||
       !aligned16(store->val_v)))
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  if (k > c->S) return TD_ERR_INVALID_ARG;
  const int nl = layer_end - layer_begin;
  StoreDev sd;
  sd.master_k = static_cast<uint16_t*>(store->master_k);
  sd.master_v = static_cast<uint16_t*>(store->master_v);
  sd.rowptr = store->rowptr;
  sd.block_idx = store->block_idx;
  sd.val_k = static_cast<uint16_t*>(store->val_k);
  sd.val_v = static_cast<uint16_t*>(store->val_v);
  sd.slot = store->slot;
  sd.capacity = store->capacity_blocks;
  sd.nl = nl;
  EncodeScratch sc;
  sc.selbits = c->d_selbits;
  sc.firstrank = c->d_firstrank;
  sc.mask = c->d_mask;
  sc.cand = c->d_cand;
  sc.word_prefix = c->d_wprefix;
  sc.agent_prefix = c->d_aprefix;
  sc.flag = c->d_flag;
  sc.row_count = reinterpret_cast<int32_t*>(
      c->d_flag + static_cast<size_t>(c->N) * nl * round_dev(c).nb);
  sc.words = c->d_ints;
  sc.nbw = (round_dev(c).nb + 31) / 32;
  cudaError_t e = launch_encode(c->g, round_dev(c), master,
                                static_cast<const uint16_t*>(k_canon),
                                static_cast<const uint16_t*>(v_canon), sel, k,
                                static_cast<const uint16_t*>(k_fresh_sel),
                                static_cast<const uint16_t*>(v_fresh_sel), nl, sd, sc, c->d_err,
                                c->d_bound, st);
  if (e != cudaSuccess || note_use(c, st) != TD_OK) return TD_ERR_CUDA;
  store->layer_begin = layer_begin;
  store->layer_end = layer_end;
  if (nnz_out) {
    int64_t* h = c->h_words;
    if (cudaMemcpyAsync(h, c->d_bound, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(h + 1, store->rowptr + static_cast<int64_t>(c->N) * nl, 8,
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return TD_ERR_CUDA;
    if (h[0] > store->capacity_blocks) {
      *nnz_out = h[0];
      return TD_ERR_CAPACITY;
    }
    *nnz_out = h[1];
  }
  return TD_OK;
}

td_status td_fused_restore(td_ctx* c, const td_round* r, const td_diff_store* store,
                           const int32_t* agents, int32_t n_list, int32_t layer_begin,
                           int32_t layer_end, int32_t frame, const td_paged* pool,
                           void* stream) {
  if (!c || !same_device(c) || !store || (n_list > 0 && !agents) || n_list < 0 ||
      (frame != 0 && frame != 1))
    return TD_ERR_INVALID_ARG;
  if (!store->master_k || !store->master_v || !store->slot || !aligned16(store->master_k) ||
      !aligned16(store->master_v))
    return TD_ERR_INVALID_ARG;
  if (layer_begin < store->layer_begin || layer_end > store->layer_end ||
      layer_begin >= layer_end || store->layer_begin < 0 ||
      store->layer_end > c->shape.n_layers)
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  for (int x = 0; x < n_list; ++x)
    if (agents[x] < 0 || agents[x] >= c->N) return TD_ERR_INVALID_ARG;
  PoolDev pd;
  if ((s = pool_dev(c, r, pool, &pd)) != TD_OK) return s;
  StoreDev sd;
  sd.master_k = static_cast<uint16_t*>(store->master_k);
  sd.master_v = static_cast<uint16_t*>(store->master_v);
  sd.rowptr = store->rowptr;
  sd.block_idx = store->block_idx;
  sd.val_k = static_cast<uint16_t*>(store->val_k);
  sd.val_v = static_cast<uint16_t*>(store->val_v);
  sd.slot = store->slot;
  sd.capacity = store->capacity_blocks;
  sd.nl = store->layer_end - store->layer_begin;
  const RoundDev rd = round_dev(c);
  for (int x0 = 0; x0 < n_list; x0 += kMaxListAgents) {
    AgentList al;
    al.n = n_list - x0 < kMaxListAgents ? n_list - x0 : kMaxListAgents;
    for (int x = 0; x < al.n; ++x) al.a[x] = agents[x0 + x];
    cudaError_t e = launch_restore(c->g, rd, pd, sd, al, layer_begin, store->layer_begin,
                                   layer_end - layer_begin, frame, c->d_err, st);
    if (e != cudaSuccess) return TD_ERR_CUDA;
  }
  return note_use(c, st);
}

td_status td_materialise_mirror(td_ctx* c, const td_round* r, const td_diff_store* store,
                                int32_t agent, int32_t layer_begin, int32_t layer_end,
                                void* dense_k, void* dense_v, void* stream) {
  if (!c || !same_device(c) || !store || !dense_k || !dense_v || !aligned16(dense_k) ||
      !aligned16(dense_v))
    return TD_ERR_INVALID_ARG;
  if (!store->master_k || !store->master_v || !store->slot || !aligned16(store->master_k) ||
      !aligned16(store->master_v))
    return TD_ERR_INVALID_ARG;
  if (layer_begin < store->layer_begin || layer_end > store->layer_end ||
      layer_begin >= layer_end || store->layer_begin < 0 ||
      store->layer_end > c->shape.n_layers)
    return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  td_status s = prepare_round(c, r, st);
  if (s != TD_OK) return s;
  if (agent < 0 || agent >= c->N) return TD_ERR_INVALID_ARG;
  StoreDev sd;
  sd.master_k = static_cast<uint16_t*>(store->master_k);
  sd.master_v = static_cast<uint16_t*>(store->master_v);
  sd.rowptr = store->rowptr;
  sd.block_idx = store->block_idx;
  sd.val_k = static_cast<uint16_t*>(store->val_k);
  sd.val_v = static_cast<uint16_t*>(store->val_v);
  sd.slot = store->slot;
  sd.capacity = store->capacity_blocks;
  sd.nl = store->layer_end - store->layer_begin;
  if (launch_materialise(c->g, round_dev(c), sd, agent, layer_begin - store->layer_begin,
                         layer_end - layer_begin, static_cast<uint16_t*>(dense_k),
                         static_cast<uint16_t*>(dense_v), c->d_err, st) != cudaSuccess)
    return TD_ERR_CUDA;
  return note_use(c, st);
}

td_status td_fused_attention(td_ctx* c, const td_round* r, const td_diff_store* store,
                             const td_paged* pool, const int32_t* agents, int32_t n_list,
                             int32_t layer_begin, int32_t layer_end, const void* q,
                             int32_t n_q_heads, float scale, float* out, float* lse,
                             void* stream) {
  if (!store) return TD_ERR_INVALID_ARG;
  return run_attention(c, r, store, pool, agents, n_list, layer_begin, layer_end, q, n_q_heads,
                       scale, out, lse, stream);
}

td_status td_paged_attention(td_ctx* c, const td_round* r, const td_paged* pool,
                             const int32_t* agents, int32_t n_list, int32_t layer_begin,
                             int32_t layer_end, const void* q, int32_t n_q_heads, float scale,
                             float* out, float* lse, void* stream) {
  return run_attention(c, r, nullptr, pool, agents, n_list, layer_begin, layer_end, q, n_q_heads,
                       scale, out, lse, stream);
}

td_status td_inject_attention_wait_fault(td_ctx* c, uint32_t bytes) {
  if (!c) return TD_ERR_INVALID_ARG;
  c->attn_tx_pad = bytes;
  return TD_OK;
}

td_status td_get_error(td_ctx* c, void* stream, uint32_t* bits_out) {
  if (!c || !same_device(c)) return TD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* h = reinterpret_cast<uint32_t*>(c->h_words);
  if (cudaMemcpyAsync(h, c->d_err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(c->d_err, 0, 4, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return TD_ERR_CUDA;
  const uint32_t bits = *h;
  if (bits_out) *bits_out = bits;
  for (int code = 1; code < 32; ++code)
    if (bits & (1u << code)) return static_cast<td_status>(code);
  return TD_OK;
}

}  // extern "C"
