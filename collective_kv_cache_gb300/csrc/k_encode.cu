// k_encode.cu - stage 3b: Master-Mirror block-sparse encoding (TokenDance review [R],
// Summary Method (3): the Master keeps a full cache, every other agent records only the
// indices and values of the blocks where it differs; Figure 8; §2b item 2: one
// (indices, values) record per Mirror per layer).
//
// Only blocks that hold a selected token of the Mirror or of the Master can differ (every
// other token of both is the canonical K/V itself), so the candidate blocks of Mirror i
// are mask_i | mask_master. Their number per layer is known before any K/V is read, which
// gives every candidate block a fixed place in the store:
//   prep    per agent: a 16-bit mask of its selected tokens in each diff block, the rank
//           of the block's first selected token, and its block bitmask
//   cand    candidate masks, per-word and per-agent prefix counts, the bound
//           nl * sum_i |cand_i|, master sanity
//   main    one CTA per (layer, 16-token block, K or V, part): reads its canonical data
//           once, builds the Master's (recomputed K turned back by R(-off)) and writes it,
//           then for each candidate Mirror builds its half-tile, writes it at its
//           candidate place and ORs "differs" into the block's flag, one atomic per warp;
//           the warp that sets a flag first counts the record in its row. No barriers.
//   rows    exclusive prefix sum of the per-(agent, layer) record counts (rowptr)
//   index   block indices and the (agent, layer, block) -> record slot map
//   fixup   only when some candidate equalled the Master's block: rewrite the kept
//           blocks whose record moved (recomputed from the inputs, never copied)
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
  uint32_t* err;
};

__global__ void __launch_bounds__(1024) enc_prep_kernel(EncArgs a) {
  extern __shared__ unsigned smask[];
  const int i = blockIdx.x;
  const int S = a.rd.S, nb = a.rd.nb, k = a.k, nbw = a.sc.nbw;
  uint32_t* bits = a.sc.selbits + static_cast<int64_t>(i) * nb;
  int32_t* first = a.sc.firstrank + static_cast<int64_t>(i) * nb;
  const int32_t* sel = a.sel + static_cast<int64_t>(i) * k;
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
    const int b = t / kDiffBlock;
    atomicOr(&bits[b], 1u << (t - b * kDiffBlock));
    if (prev < 0 || prev / kDiffBlock != b) first[b] = r;
    atomicOr(&smask[b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) a.sc.mask[i * nbw + w] = smask[w];
}

__global__ void __launch_bounds__(1024) enc_cand_kernel(EncArgs a, const int32_t* master) {
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
  }
  __syncthreads();
  const int m = s_m;
  if (m < 0) return;
  for (int x = threadIdx.x; x < N * nbw; x += blockDim.x) {
    const int i = x / nbw, w = x - (x / nbw) * nbw;
    a.sc.cand[x] = i == m ? 0u : (a.sc.mask[x] | a.sc.mask[m * nbw + w]);
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
    *a.sc.need_fixup = 0;
  }
}

__device__ __forceinline__ int64_t cand_place(const EncArgs& a, int i, int li, int b) {
  const int nbw = a.sc.nbw;
  const int64_t ap0 = a.sc.agent_prefix[i], ap1 = a.sc.agent_prefix[i + 1];
  const unsigned word = a.sc.cand[i * nbw + (b >> 5)];
  const unsigned below = (b & 31) ? (word & ((1u << (b & 31)) - 1u)) : 0u;
  return ap0 * a.nl + static_cast<int64_t>(li) * (ap1 - ap0) +
         a.sc.word_prefix[i * nbw + (b >> 5)] + __popc(below);
}

// Per-thread items of one half-tile (K or V) of a (layer, block) tile.
template <int kItems>
struct HalfTile {
  int tl[kItems];     // token within the block
  int e0[kItems];
  int f0[kItems];
  int blk[kItems];
  bool live[kItems];  // token < S
  bool pad[kItems];   // item of the block's tail (token >= S): zeros in the store
  uint4 c0[kItems], c1[kItems];  // canonical pair-vector
};

template <int kItems>
__device__ __forceinline__ void load_half(const EncArgs& a, int li, int t0, int kv, int q0,
                                          HalfTile<kItems>& h) {
  const int n_items = kDiffBlock * a.g.vpt;
  const uint16_t* src = kv == 0 ? a.kc : a.vc;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = q0 + threadIdx.x + r * blockDim.x;
    const Item it = item_of(a.g, q < n_items ? q : 0);
    const int t = t0 + it.tok;
    h.tl[r] = it.tok;
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
  if (!((sbits >> h.tl[r]) & 1u)) return;
  const int rk = first + __popc(sbits & ((1u << h.tl[r]) - 1u));
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
                  (rec * kDiffBlock + h.tl[r]) * a.g.E;
  st16(dst + h.e0[r], x0);
  st16(dst + h.e0[r] + a.g.half, x1);
}

template <int kItems>
__global__ void __launch_bounds__(256, 3) enc_main_kernel(EncArgs a, int tiles_per_layer) {
  const int m = *a.m_ok;
  if (m < 0) return;
  const int over = *a.over;
  const Unit un = unit_of(a.g, blockIdx.x, tiles_per_layer);
  const int kv = un.kv, li = un.li, b = un.b;
  const int t0 = b * kDiffBlock;
  const int N = a.rd.N, nb = a.rd.nb, nbw = a.sc.nbw;
  const int lane = threadIdx.x & 31;

  HalfTile<kItems> h;
  load_half<kItems>(a, li, t0, kv, un.q0, h);

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

  // per-agent facts of this block, one chunk of agents at a time
  __shared__ int64_t s_place[kAgentChunk];   // candidate place, -1 = not a candidate
  __shared__ unsigned s_bits[kAgentChunk];
  __shared__ int s_first[kAgentChunk];
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int c0 = 0; c0 < N; c0 += kAgentChunk) {
    const int n = min(kAgentChunk, N - c0);
    if (c0 > 0) __syncthreads();
    for (int x = threadIdx.x; x < n; x += blockDim.x) {
      const int i = c0 + x;
      const unsigned word = a.sc.cand[i * nbw + (b >> 5)];
      const bool is_cand = (word >> (b & 31)) & 1u;
      const unsigned ibits = is_cand ? a.sc.selbits[static_cast<int64_t>(i) * nb + b] : 0u;
      s_place[x] = is_cand ? cand_place(a, i, li, b) : -1;
      s_bits[x] = ibits;
      s_first[x] = ibits ? a.sc.firstrank[static_cast<int64_t>(i) * nb + b] : 0;
    }
    __syncthreads();
    for (int x = 0; x < n; ++x) {
      const int64_t rec = s_place[x];
      if (rec < 0) continue;                       // uniform across the CTA
      const int i = c0 + x;
      const unsigned ibits = s_bits[x];
      const int ifirst = s_first[x];
      bool d = false;
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (h.live[r]) {
          uint4 x0, x1;
          agent_item<kItems>(a, i, li, kv, ibits, ifirst, h, r, x0, x1);
          d |= neq16(x0, m0[r]) | neq16(x1, m1[r]);
          if (!over) store_item<kItems>(a, kv, rec, h, r, x0, x1);
        } else if (h.pad[r] && !over) {
          store_item<kItems>(a, kv, rec, h, r, z, z);
        }
      }
      if (__any_sync(0xFFFFFFFFu, d) && lane == 0) {
        const int64_t f = (static_cast<int64_t>(i) * a.nl + li) * nb + b;
        if (atomicOr(a.sc.flag + f, 1u) == 0u)
          atomicAdd(a.sc.row_count + static_cast<int64_t>(i) * a.nl + li, 1);
      }
    }
  }
}

// Exclusive prefix sum of the per-(agent, layer) record counts -> rowptr.
__global__ void __launch_bounds__(1024) enc_rows_kernel(EncArgs a) {
  __shared__ long long wsum[32];
  if (*a.m_ok < 0) return;
  const int R = a.rd.N * a.nl;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int per = (R + blockDim.x - 1) / blockDim.x;
  const int r0 = threadIdx.x * per, r1 = min(R, r0 + per);
  long long local = 0;
  for (int r = r0; r < r1; ++r) local += a.sc.row_count[r];
  long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  long long before = 0;
  for (int w = 0; w < wid; ++w) before += wsum[w];
  long long run = before + incl - local;
  for (int r = r0; r < r1; ++r) {
    a.store.rowptr[r] = run;
    run += a.sc.row_count[r];
  }
  if (threadIdx.x == blockDim.x - 1) {
    long long total = 0;
    for (int w = 0; w < nw; ++w) total += wsum[w];
    a.store.rowptr[R] = total;
    if (!*a.over && total != *a.bound) *a.sc.need_fixup = 1;
  }
}

// Block indices and the slot map; one warp per (agent, layer) row.
__global__ void __launch_bounds__(256) enc_index_kernel(EncArgs a) {
  if (*a.m_ok < 0 || *a.over) return;
  const int R = a.rd.N * a.nl, nb = a.rd.nb;
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= R) return;
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

// Rewrites the kept blocks whose record is not at their candidate place (only when some
// candidate turned out equal to the Master's block). Grid-stride over (tile, K/V).
template <int kItems>
__global__ void __launch_bounds__(256) enc_fixup_kernel(EncArgs a, int tiles_per_layer) {
  if (*a.sc.need_fixup == 0) return;
  const int m = *a.m_ok;
  if (m < 0) return;
  const int nb = a.rd.nb;
  const int64_t units = static_cast<int64_t>(tiles_per_layer) * a.nl * 2 * parts_per_tile(a.g);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const Unit un = unit_of(a.g, u, tiles_per_layer);
    const int kv = un.kv, li = un.li, b = un.b;
    HalfTile<kItems> h;
    load_half<kItems>(a, li, b * kDiffBlock, kv, un.q0, h);
    for (int i = 0; i < a.rd.N; ++i) {
      if (i == m) continue;
      const int s = a.store.slot[(static_cast<int64_t>(i) * a.nl + li) * nb + b];
      if (s < 0 || s == cand_place(a, i, li, b)) continue;
      const unsigned ibits = a.sc.selbits[static_cast<int64_t>(i) * nb + b];
      const int ifirst = ibits ? a.sc.firstrank[static_cast<int64_t>(i) * nb + b] : 0;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (h.live[r]) {
          uint4 x0, x1;
          agent_item<kItems>(a, i, li, kv, ibits, ifirst, h, r, x0, x1);
          store_item<kItems>(a, kv, s, h, r, x0, x1);
        } else if (h.pad[r]) {
          store_item<kItems>(a, kv, s, h, r, z, z);
        }
      }
    }
  }
}

template <int kItems>
static cudaError_t run_tiles(const EncArgs& a, int threads, cudaStream_t st) {
  const int tpl = a.rd.nb;
  const int64_t units = static_cast<int64_t>(tpl) * a.nl * 2 * parts_per_tile(a.g);
  enc_main_kernel<kItems><<<static_cast<unsigned>(units), threads, 0, st>>>(a, tpl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  enc_rows_kernel<<<1, 1024, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.rd.N) * a.nl;
  enc_index_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t fix_grid = units < 1216 ? units : 1216;
  enc_fixup_kernel<kItems><<<static_cast<unsigned>(fix_grid), threads, 0, st>>>(a, tpl);
  return cudaGetLastError();
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
  a.m_ok = sc.need_fixup + 1;  // the context lays these three ints out after need_fixup
  a.over = sc.need_fixup + 2;
  a.bound = bound_dev;
  a.err = err;
  if (nl <= 0) return cudaSuccess;
  // flags and row counts start at zero (one contiguous region)
  const size_t flag_words = static_cast<size_t>(rd.N) * nl * rd.nb;
  cudaError_t e = cudaMemsetAsync(sc.flag, 0, (flag_words + static_cast<size_t>(rd.N) * nl) * 4, st);
  if (e != cudaSuccess) return e;
  enc_prep_kernel<<<rd.N, 1024, sc.nbw * sizeof(unsigned), st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  enc_cand_kernel<<<1, 1024, 0, st>>>(a, master);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int threads = tile_threads(g);
  if (tile_items(g) == 1) return run_tiles<1>(a, threads, st);
  return run_tiles<2>(a, threads, st);
}

}  // namespace td
