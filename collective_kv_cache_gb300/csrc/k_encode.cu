// k_encode.cu - stage 3b: Master-Mirror block-sparse encoding (TokenDance review [R],
// Summary Method (3): the Master keeps a full cache, every other agent records only the
// indices and values of the blocks where it differs; Figure 8; §2b item 2: one
// (indices, values) record per Mirror per layer).
//
// Only blocks that hold a selected token of the Mirror or of the Master can differ (every
// other token of both is the canonical K/V itself), so the candidate blocks of Mirror i
// are mask_i | mask_master. Their number per layer is known before any K/V is read, which
// gives every candidate block a fixed place in the store. Four launches:
//   prep    one CTA per agent: zeroes the agent's flags and record counts, builds a
//           mask of its selected tokens in each diff block (16 or 32 bits), the rank of the
//           block's first selected token and its block bitmask; the CTA that finishes
//           last (a self-resetting counter; no CTA waits) builds the candidate masks, the
//           per-word and per-agent prefix counts, the bound nl * sum_i |cand_i|, and
//           checks the master
//   main    one CTA per (layer, 16-token tile, K or V, part), the tiles covering whole
//           diff blocks (a 32-token block is two tiles): reads its canonical data
//           once, builds the Master's (recomputed K turned back by R(-off)) and writes it,
//           then for each candidate Mirror builds its data, writes it at its candidate
//           place and, where it differs (one warp vote), ORs the block's flag without
//           waiting for the result. One CTA per block writes the slot map and block
//           indices of the common case (every candidate kept);
//   rows    each (agent, layer) row's record count from its flags, one warp a row over
//           as many CTAs as the rows need;
//   fixup   every CTA takes the prefix of the counts (CTA 0 writes rowptr); only when
//           some candidate equalled the Master's block does it compact the slot map and
//           indices and rewrite the kept blocks whose record moved (recomputed from the
//           inputs, never copied); otherwise it returns at once.
// No Mirror is built densely; in the common case the inputs are read once.
#include "td_device.cuh"

namespace td {

struct EncArgs {
  Geom g;
  RoundDev rd;
  const uint16_t* kc;   // [nl][S][E]
  const uint16_t* vc;
  const int32_t* sel;   // [N][k]
  int k;
  const uint16_t* kf;   // [N][nl][k][E]
  const uint16_t* vf;
  int nl;
  StoreDev store;
  EncodeScratch sc;
  int32_t* m_ok;        // sanitized master (-1 = invalid)
  int32_t* over;        // bound exceeds capacity
  int64_t* bound;
  int* prep_done;       // CTAs of prep finished (self-resetting)
  uint32_t* err;
};

// Candidate masks, prefix counts, bound and master check (run by the last prep CTA).
__device__ void build_candidates(const EncArgs& a, const int32_t* master) {
  const int N = a.rd.N, nbw = a.sc.nbw;
  __shared__ int s_m;
  if (threadIdx.x == 0) {
    int m = *master;
    if (m < 0 || m >= N) {
      atomicOr(a.err, err_bit(TD_ERR_INVALID_ARG));
      m = -1;
    }
    s_m = m;
    *a.m_ok = m;
    *a.over = 0;
  }
  __syncthreads();
  const int m = s_m;
  if (m < 0) return;
  for (int x = threadIdx.x; x < N * nbw; x += blockDim.x) {
    const int i = x / nbw, w = x - (x / nbw) * nbw;
    a.sc.cand[x] = i == m ? 0u : (__ldcg(a.sc.mask + x) | __ldcg(a.sc.mask + m * nbw + w));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nbw; ++w) {
      a.sc.word_prefix[i * nbw + w] = run;
      run += __popc(a.sc.cand[i * nbw + w]);
    }
    a.sc.word_prefix[N * nbw + i] = run;  // per-agent count, consumed below
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t run = 0;
    for (int i = 0; i < N; ++i) {
      a.sc.agent_prefix[i] = run;
      run += a.sc.word_prefix[N * nbw + i];
    }
    a.sc.agent_prefix[N] = run;
    const int64_t bound = run * a.nl;
    *a.bound = bound;
    const int over = bound > a.store.capacity ? 1 : 0;
    *a.over = over;
    if (over) atomicOr(a.err, err_bit(TD_ERR_CAPACITY));
  }
}

__global__ void __launch_bounds__(1024) enc_prep_kernel(EncArgs a, const int32_t* master) {
  extern __shared__ unsigned smask[];
  __shared__ int s_last;
  // once every earlier kernel has finished (so the canonical rows are final), the main
  // kernel may start reading them while prep runs
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int S = a.rd.S, nb = a.rd.nb, k = a.k, nbw = a.sc.nbw;
  uint32_t* bits = a.sc.selbits + static_cast<int64_t>(i) * nb;
  int32_t* first = a.sc.firstrank + static_cast<int64_t>(i) * nb;
  const int32_t* sel = a.sel + static_cast<int64_t>(i) * k;
  uint32_t* flags = a.sc.flag + static_cast<int64_t>(i) * a.nl * nb;
  for (int x = threadIdx.x; x < a.nl * nb; x += blockDim.x) flags[x] = 0u;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) bits[b] = 0u;
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) smask[w] = 0u;
  __syncthreads();
  for (int r = threadIdx.x; r < k; r += blockDim.x) {
    const int t = __ldg(sel + r);
    const int prev = r > 0 ? __ldg(sel + r - 1) : -1;
    if (t < 0 || t >= S || t <= prev) {   // rows must be ascending and in range
      atomicOr(a.err, err_bit(TD_ERR_INVALID_ARG));
      continue;
    }
    const int b = t / a.rd.B;
    atomicOr(&bits[b], 1u << (t - b * a.rd.B));
    if (prev < 0 || prev / a.rd.B != b) first[b] = r;
    atomicOr(&smask[b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) a.sc.mask[i * nbw + w] = smask[w];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.prep_done, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (!s_last) return;                        // uniform across the CTA
  __threadfence();
  if (threadIdx.x == 0) *a.prep_done = 0;     // ready for the next call
  build_candidates(a, master);
}

__device__ __forceinline__ int64_t cand_place(const EncArgs& a, int i, int li, int b) {
  const int nbw = a.sc.nbw;
  const int64_t ap0 = a.sc.agent_prefix[i], ap1 = a.sc.agent_prefix[i + 1];
  const unsigned word = a.sc.cand[i * nbw + (b >> 5)];
  const unsigned below = (b & 31) ? (word & ((1u << (b & 31)) - 1u)) : 0u;
  return ap0 * a.nl + static_cast<int64_t>(li) * (ap1 - ap0) +
         a.sc.word_prefix[i * nbw + (b >> 5)] + __popc(below);
}

// Exclusive prefix sum of the per-(agent, layer) record counts, in chunks of kPrefixPer
// rows a thread whose counts are all loaded at once; written to rowptr when `write`.
// Returns the total. Every thread of the CTA calls it.
constexpr int kPrefixPer = 8;

__device__ long long rows_prefix(const EncArgs& a, bool write) {
  __shared__ long long wsum[32];
  const int R = a.rd.N * a.nl;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long carry = 0;
  for (int c0 = 0; c0 < R; c0 += blockDim.x * kPrefixPer) {
    const int r0 = c0 + threadIdx.x * kPrefixPer;
    int cnt[kPrefixPer];
    long long local = 0;
#pragma unroll
    for (int q = 0; q < kPrefixPer; ++q) {
      cnt[q] = r0 + q < R ? __ldcg(a.sc.row_count + r0 + q) : 0;
      local += cnt[q];
    }
    long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < nw; ++w) {
      if (w < wid) before += wsum[w];
      total += wsum[w];
    }
    long long run = carry + before + incl - local;
    if (write) {
#pragma unroll
      for (int q = 0; q < kPrefixPer; ++q) {
        if (r0 + q < R) a.store.rowptr[r0 + q] = run;
        run += cnt[q];
      }
    }
    carry += total;
    __syncthreads();   // wsum is rewritten by the next chunk
  }
  if (write && threadIdx.x == 0) a.store.rowptr[R] = carry;
  return carry;
}

// Per-thread items of one half-tile (K or V) of a (layer, 16-token tile) unit.
template <int kItems>
struct HalfTile {
  int tl[kItems];     // token within the tile
  int tb[kItems];     // row within the diff block (the tile's first row tb0 + tl)
  int e0[kItems];
  int f0[kItems];
  int blk[kItems];
  bool live[kItems];  // token < S
  bool pad[kItems];   // item of the block's tail (token >= S): zeros in the store
  uint4 c0[kItems], c1[kItems];  // canonical pair-vector
};

template <int kItems>
__device__ __forceinline__ void load_half(const EncArgs& a, int li, int t0, int tb0, int kv,
                                          int q0, HalfTile<kItems>& h) {
  const int n_items = kTile * a.g.vpt;
  const uint16_t* src = kv == 0 ? a.kc : a.vc;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = q0 + threadIdx.x + r * blockDim.x;
    const Item it = item_of(a.g, q < n_items ? q : 0);
    const int t = t0 + it.tok;
    h.tl[r] = it.tok;
    h.tb[r] = tb0 + it.tok;
    h.e0[r] = it.e0;
    h.f0[r] = it.f0;
    h.live[r] = q < n_items && t < a.rd.S;
    h.pad[r] = q < n_items && t >= a.rd.S;
    h.blk[r] = 0;
    h.c0[r] = h.c1[r] = make_uint4(0u, 0u, 0u, 0u);
    if (h.live[r]) {
      const int64_t row = (static_cast<int64_t>(li) * a.rd.S + t) * a.g.E;
      h.c0[r] = ldg16(src + row + it.e0);
      h.c1[r] = ldg16(src + row + it.e0 + a.g.half);
      if (kv == 0) h.blk[r] = __ldg(a.rd.tok_block + t);
    }
  }
}

// Agent `ag`'s canonical-frame value of item r: its recomputed K turned back by R(-off)
// (or its recomputed V) when the item's token is selected, the canonical value otherwise.
template <int kItems>
__device__ __forceinline__ void agent_item(const EncArgs& a, int ag, int li, int kv,
                                           unsigned sbits, int first, const HalfTile<kItems>& h,
                                           int r, uint4& x0, uint4& x1) {
  x0 = h.c0[r];
  x1 = h.c1[r];
  if (!((sbits >> h.tb[r]) & 1u)) return;
  const int rk = first + __popc(sbits & ((1u << h.tb[r]) - 1u));
  const int64_t row = ((static_cast<int64_t>(ag) * a.nl + li) * a.k + rk) * a.g.E;
  if (kv == 0) {
    const uint4 fa = ldg16(a.kf + row + h.e0[r]);
    const uint4 fb = ldg16(a.kf + row + h.e0[r] + a.g.half);
    const int64_t toff = static_cast<int64_t>(ag * a.rd.M + h.blk[r]) * a.g.half + h.f0[r];
    rotate_pairs<true>(fa, fb, a.rd.cos_t + toff, a.rd.sin_t + toff, x0, x1);
  } else {
    x0 = ldg16(a.vf + row + h.e0[r]);
    x1 = ldg16(a.vf + row + h.e0[r] + a.g.half);
  }
}

template <int kItems>
__device__ __forceinline__ void store_item(const EncArgs& a, int kv, int64_t rec,
                                           const HalfTile<kItems>& h, int r, const uint4& x0,
                                           const uint4& x1) {
  uint16_t* dst = (kv == 0 ? a.store.val_k : a.store.val_v) +
                  (rec * a.rd.B + h.tb[r]) * a.g.E;
  st16(dst + h.e0[r], x0);
  st16(dst + h.e0[r] + a.g.half, x1);
}

constexpr int kStageDepth = 3;   // candidates in flight per thread

// Stage, for candidate agent `ag`, the recomputed data of this thread's selected items:
// slot [depth][0/1][item][thread] (each thread touches only its own 16-byte cells).
template <int kItems>
__device__ __forceinline__ void stage_candidate(const EncArgs& a, int ag, int li, int kv,
                                                unsigned sbits, int first,
                                                const HalfTile<kItems>& h, uint4* slot) {
  const uint16_t* src = kv == 0 ? a.kf : a.vf;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    if (!h.live[r] || !((sbits >> h.tb[r]) & 1u)) continue;
    const int rk = first + __popc(sbits & ((1u << h.tb[r]) - 1u));
    const uint16_t* row = src + ((static_cast<int64_t>(ag) * a.nl + li) * a.k + rk) * a.g.E;
    cp_async16(slot + (0 * kItems + r) * blockDim.x + threadIdx.x, row + h.e0[r]);
    cp_async16(slot + (1 * kItems + r) * blockDim.x + threadIdx.x, row + h.e0[r] + a.g.half);
  }
  cp_async_commit();
}

// Candidate agent `ag`'s value of item r from its staged data (K turned back by R(-off)).
template <int kItems>
__device__ __forceinline__ void staged_item(const EncArgs& a, int ag, int kv, unsigned sbits,
                                            const HalfTile<kItems>& h, int r,
                                            const uint4* slot, uint4& x0, uint4& x1) {
  x0 = h.c0[r];
  x1 = h.c1[r];
  if (!((sbits >> h.tb[r]) & 1u)) return;
  const uint4 fa = slot[(0 * kItems + r) * blockDim.x + threadIdx.x];
  const uint4 fb = slot[(1 * kItems + r) * blockDim.x + threadIdx.x];
  if (kv == 0) {
    const int64_t toff = static_cast<int64_t>(ag * a.rd.M + h.blk[r]) * a.g.half + h.f0[r];
    rotate_pairs<true>(fa, fb, a.rd.cos_t + toff, a.rd.sin_t + toff, x0, x1);
  } else {
    x0 = fa;
    x1 = fb;
  }
}

// 4- and 8-byte asynchronous copies (through L1), for the per-agent facts.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(gmem) : "memory");
}

template <int kItems>
__global__ void __launch_bounds__(256, 3) enc_main_kernel(EncArgs a, int tiles_per_layer) {
  const Unit un = unit_of(a.g, blockIdx.x, tiles_per_layer);
  const int kv = un.kv, li = un.li;
  const int t0 = un.b * kTile;
  const int b = t0 / a.rd.B;                 // the tile's diff block
  const int tb0 = t0 - b * a.rd.B;           // the tile's first row within it
  const int N = a.rd.N, nb = a.rd.nb, nbw = a.sc.nbw;
  const int lane = threadIdx.x & 31;

  pdl_trigger();
  // the raw per-agent facts of this block for one chunk of agents, copied in by the first
  // warp once prep has finished
  __shared__ unsigned s_word[kAgentChunk], s_sb[kAgentChunk];
  __shared__ int s_fr[kAgentChunk], s_wp[kAgentChunk];
  __shared__ int64_t s_ap[kAgentChunk + 1];
  auto fetch_facts = [&](int c0, int n) {
    for (int x = lane; x < n; x += 32) {
      const int i = c0 + x;
      cp_async4(&s_word[x], a.sc.cand + i * nbw + (b >> 5));
      cp_async4(&s_sb[x], a.sc.selbits + static_cast<int64_t>(i) * nb + b);
      cp_async4(&s_fr[x], a.sc.firstrank + static_cast<int64_t>(i) * nb + b);
      cp_async4(&s_wp[x], a.sc.word_prefix + i * nbw + (b >> 5));
      cp_async8(&s_ap[x], a.sc.agent_prefix + i);
    }
    if (lane == 0) cp_async8(&s_ap[n], a.sc.agent_prefix + c0 + n);
    cp_async_commit();
  };
  // the canonical rows are inputs, final once prep has started: read before it finishes
  HalfTile<kItems> h;
  load_half<kItems>(a, li, t0, tb0, kv, un.q0, h);
  pdl_wait();
  if (threadIdx.x < 32) fetch_facts(0, min(kAgentChunk, N));
  const int m = *a.m_ok;
  if (m < 0) {
    cp_async_wait<0>();
    return;
  }
  const int over = *a.over;
  // the Master's half-tile, written dense
  const unsigned mbits = a.sc.selbits[static_cast<int64_t>(m) * nb + b];
  const int mfirst = mbits ? a.sc.firstrank[static_cast<int64_t>(m) * nb + b] : 0;
  uint4 m0[kItems], m1[kItems];
  uint16_t* mdst = kv == 0 ? a.store.master_k : a.store.master_v;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    if (!h.live[r]) continue;
    agent_item<kItems>(a, m, li, kv, mbits, mfirst, h, r, m0[r], m1[r]);
    const int64_t row = (static_cast<int64_t>(li) * a.rd.S + t0 + h.tl[r]) * a.g.E;
    st16(mdst + row + h.e0[r], m0[r]);
    st16(mdst + row + h.e0[r] + a.g.half, m1[r]);
  }

  const bool designated = kv == 0 && un.q0 == 0 && tb0 == 0;  // one CTA per block: slot/index
  // per-agent facts of this block, one chunk of agents at a time
  __shared__ int64_t s_place[kAgentChunk];   // candidate place, -1 = not a candidate
  __shared__ unsigned s_bits[kAgentChunk];
  __shared__ int s_first[kAgentChunk];
  __shared__ int s_list[kAgentChunk];        // the chunk's candidates, in agent order
  __shared__ int s_nc;
  extern __shared__ uint4 s_stage[];         // [kStageDepth][2][kItems][blockDim]
  const int slot_cells = 2 * kItems * blockDim.x;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int c0 = 0; c0 < N; c0 += kAgentChunk) {
    const int n = min(kAgentChunk, N - c0);
    if (c0 > 0) {
      __syncthreads();
      if (threadIdx.x < 32) fetch_facts(c0, n);
    }
    if (threadIdx.x < 32) {
      // the first warp alone: the chunk's candidate places, then the candidates compacted
      // in agent order (no staging copy is pending here: the previous chunk drained them)
      cp_async_wait<0>();
      __syncwarp();
      for (int x = threadIdx.x; x < n; x += 32) {
        const int i = c0 + x;
        const unsigned word = s_word[x];
        const int64_t ap0 = s_ap[x], ap1 = s_ap[x + 1];
        const bool is_cand = (word >> (b & 31)) & 1u;
        const unsigned below = (b & 31) ? (word & ((1u << (b & 31)) - 1u)) : 0u;
        const int64_t place = is_cand ? ap0 * a.nl + static_cast<int64_t>(li) * (ap1 - ap0) +
                                            s_wp[x] + __popc(below)
                                      : -1;
        const unsigned ibits = is_cand ? s_sb[x] : 0u;
        s_place[x] = place;
        s_bits[x] = ibits;
        s_first[x] = ibits ? s_fr[x] : 0;
        if (designated && !over) {   // slot map and index of the common case
          a.store.slot[(static_cast<int64_t>(i) * a.nl + li) * nb + b] =
              static_cast<int32_t>(place);
          if (place >= 0) a.store.block_idx[place] = b;
        }
      }
      __syncwarp();
      int nc = 0;
      for (int x0 = 0; x0 < n; x0 += 32) {
        const int x = x0 + threadIdx.x;
        const bool c = x < n && s_place[x] >= 0;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, c);
        if (c) s_list[nc + __popc(bal & ((1u << threadIdx.x) - 1u))] = x;
        nc += __popc(bal);
      }
      if (threadIdx.x == 0) s_nc = nc;
    }
    __syncthreads();
    const int nc = s_nc;
    // pipeline: candidates j+1 .. j+depth-1 are being staged while j is built and stored
#pragma unroll
    for (int j = 0; j < kStageDepth - 1; ++j) {
      if (j < nc) {
        const int x = s_list[j];
        stage_candidate<kItems>(a, c0 + x, li, kv, s_bits[x], s_first[x], h,
                                s_stage + j * slot_cells);
      } else {
        cp_async_commit();
      }
    }
    for (int j = 0; j < nc; ++j) {
      const int jn = j + kStageDepth - 1;
      if (jn < nc) {
        const int xn = s_list[jn];
        stage_candidate<kItems>(a, c0 + xn, li, kv, s_bits[xn], s_first[xn], h,
                                s_stage + (jn % kStageDepth) * slot_cells);
      } else {
        cp_async_commit();
      }
      cp_async_wait<kStageDepth - 1>();           // candidate j has landed (this thread)
      const int x = s_list[j];
      const int i = c0 + x;
      const int64_t rec = s_place[x];
      const unsigned ibits = s_bits[x];
      const uint4* slot = s_stage + (j % kStageDepth) * slot_cells;
      bool d = false;
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (h.live[r]) {
          uint4 x0, x1;
          staged_item<kItems>(a, i, kv, ibits, h, r, slot, x0, x1);
          d |= neq16(x0, m0[r]) | neq16(x1, m1[r]);
          if (!over) store_item<kItems>(a, kv, rec, h, r, x0, x1);
        } else if (h.pad[r] && !over) {
          store_item<kItems>(a, kv, rec, h, r, z, z);
        }
      }
      // a warp whose rows differ ORs the block's flag, without waiting for the result
      if (__any_sync(0xFFFFFFFFu, d) && lane == 0)
        atomicOr(a.sc.flag + (static_cast<int64_t>(i) * a.nl + li) * nb + b, 1u);
    }
    cp_async_wait<0>();
  }
}

// After the main kernel: every (agent, layer) row's record count from its flags, one warp
// per row, spread over CTAs; the CTA that finishes last (a self-resetting counter; no CTA
// waits) takes their exclusive prefix sum -> rowptr and decides on the fix-up.
constexpr int kRowsThreads = 256;
constexpr int kRowsPerWarp = 4;   // rows a warp counts at once: their loads are all in flight

__global__ void __launch_bounds__(kRowsThreads) enc_rows_kernel(EncArgs a) {
  pdl_trigger();
  pdl_wait();
  // the flags are zeroed by prep whatever the master, so counting needs no check
  const int R = a.rd.N * a.nl, nb = a.rd.nb;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int r0 = (blockIdx.x * nw + wid) * kRowsPerWarp; r0 < R;
       r0 += gridDim.x * nw * kRowsPerWarp) {
    int cnt[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) cnt[q] = 0;
    for (int b = lane; b < nb; b += 32)
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q)
        if (r0 + q < R) cnt[q] += __ldcg(a.sc.flag + static_cast<int64_t>(r0 + q) * nb + b) != 0u;
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cnt[q] += __shfl_xor_sync(0xFFFFFFFFu, cnt[q], o);
      if (lane == 0 && r0 + q < R) a.sc.row_count[r0 + q] = cnt[q];
    }
  }
}

// The row pointers, then the fix-up. Every CTA takes the prefix of the row counts itself,
// so all agree, without waiting on one another, on whether a candidate equalled the
// Master's block (the total is below the bound); CTA 0 writes rowptr. Only then: (1)
// compact every row's slot map and block indices, warp per row; (2) rewrite each kept
// block whose final record is not its candidate place, from the inputs. The final record
// of a kept block is rowptr of its row plus the kept blocks before it, so (2) does not
// depend on (1). Grid-stride; in the common case CTA 0 writes rowptr and all return.
template <int kItems>
__global__ void __launch_bounds__(256) enc_fixup_kernel(EncArgs a, int tiles_per_layer) {
  pdl_wait();
  const int m = *a.m_ok;
  if (m < 0) return;                          // nothing was encoded: rowptr is not written
  const long long total = rows_prefix(a, blockIdx.x == 0);
  if (*a.over || total == *a.bound) return;
  // every CTA reads rowptr below: it writes the (same) values itself first
  if (blockIdx.x != 0) rows_prefix(a, true);
  __syncthreads();
  const int nb = a.rd.nb, R = a.rd.N * a.nl;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t w = warp0; w < R; w += nwarps) {
    const uint32_t* f = a.sc.flag + w * nb;
    int32_t* slot = a.store.slot + w * nb;
    int64_t run = a.store.rowptr[w];
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const bool on = b < nb && f[b] != 0u;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, on);
      const int64_t pos = run + __popc(bal & ((1u << lane) - 1u));
      if (b < nb) slot[b] = on ? static_cast<int32_t>(pos) : -1;
      if (on) a.store.block_idx[pos] = b;
      run += __popc(bal);
    }
  }
  const int64_t units = static_cast<int64_t>(tiles_per_layer) * a.nl * 2 * parts_per_tile(a.g);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const Unit un = unit_of(a.g, u, tiles_per_layer);
    const int kv = un.kv, li = un.li;
    const int t0 = un.b * kTile;
    const int b = t0 / a.rd.B;
    HalfTile<kItems> h;
    load_half<kItems>(a, li, t0, t0 - b * a.rd.B, kv, un.q0, h);
    for (int i = 0; i < a.rd.N; ++i) {
      if (i == m) continue;
      const int64_t row = static_cast<int64_t>(i) * a.nl + li;
      const uint32_t* f = a.sc.flag + row * nb;
      if (f[b] == 0u) continue;
      int64_t fin = a.store.rowptr[row];
      for (int b2 = 0; b2 < b; ++b2) fin += f[b2] != 0u;
      if (fin == cand_place(a, i, li, b)) continue;
      const unsigned ibits = a.sc.selbits[static_cast<int64_t>(i) * nb + b];
      const int ifirst = ibits ? a.sc.firstrank[static_cast<int64_t>(i) * nb + b] : 0;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (h.live[r]) {
          uint4 x0, x1;
          agent_item<kItems>(a, i, li, kv, ibits, ifirst, h, r, x0, x1);
          store_item<kItems>(a, kv, fin, h, r, x0, x1);
        } else if (h.pad[r]) {
          store_item<kItems>(a, kv, fin, h, r, z, z);
        }
      }
    }
  }
}

template <int kItems>
static cudaError_t run_tiles(const EncArgs& a, int threads, cudaStream_t st) {
  const int tpl = a.rd.nb * (a.rd.B / kTile);   // whole diff blocks: tails are zeroed
  const int64_t units = static_cast<int64_t>(tpl) * a.nl * 2 * parts_per_tile(a.g);
  // the staging ring: kStageDepth candidates x 2 vectors x kItems per thread (48 KiB at
  // 256 threads and two items); beyond the default window, so opt in (once per device)
  const size_t stage = static_cast<size_t>(kStageDepth) * 2 * kItems * threads * sizeof(uint4);
  static int opted_in_device = -1;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return cudaErrorInvalidDevice;
  if (opted_in_device != cur) {
    cudaError_t e0 = cudaFuncSetAttribute(enc_main_kernel<kItems>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kStageDepth * 2 * kItems * 256 *
                                                           sizeof(uint4)));
    if (e0 != cudaSuccess) return e0;
    opted_in_device = cur;
  }
  cudaError_t e = launch_after(enc_main_kernel<kItems>, static_cast<unsigned>(units), threads,
                               stage, st, a, tpl);
  if (e != cudaSuccess) return e;
  const int rows = a.rd.N * a.nl;
  const int per_cta = (kRowsThreads / 32) * kRowsPerWarp;
  e = launch_after(enc_rows_kernel, static_cast<unsigned>((rows + per_cta - 1) / per_cta),
                   kRowsThreads, 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_after(enc_fixup_kernel<kItems>, 152u, 256, 0, st, a, tpl);
}

cudaError_t launch_encode(const Geom& g, const RoundDev& rd, const int32_t* master,
                          const uint16_t* kc, const uint16_t* vc, const int32_t* sel, int k,
                          const uint16_t* kf, const uint16_t* vf, int nl,
                          const StoreDev& store, const EncodeScratch& sc, uint32_t* err,
                          int64_t* bound_dev, cudaStream_t st) {
  EncArgs a;
  a.g = g;
  a.rd = rd;
  a.kc = kc;
  a.vc = vc;
  a.sel = sel;
  a.k = k;
  a.kf = kf;
  a.vf = vf;
  a.nl = nl;
  a.store = store;
  a.sc = sc;
  a.m_ok = sc.words + 1;
  a.over = sc.words + 2;
  a.prep_done = sc.words + 3;
  a.bound = bound_dev;
  a.err = err;
  if (nl <= 0) return cudaSuccess;
  cudaError_t e = launch_after(enc_prep_kernel, static_cast<unsigned>(rd.N), 1024,
                               sc.nbw * sizeof(unsigned), st, a, master);
  if (e != cudaSuccess) return e;
  if (tile_items(g) == 1) return run_tiles<1>(a, tile_threads(g), st);
  return run_tiles<2>(a, tile_threads(g), st);
}

}  // namespace td
