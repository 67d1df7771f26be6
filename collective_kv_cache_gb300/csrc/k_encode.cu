// k_encode.cu - stage 3b: Master-Mirror block-sparse encoding (TokenDance review [R],
// Summary Method (3): the Master keeps a full cache, every other agent records only the
// indices and values of the blocks where it differs; Figure 8; §2b item 2: one
// (indices, values) record per Mirror per layer).
//
// Only blocks that hold a selected token of the Mirror or of the Master can differ (every
// other token of both is the canonical K/V itself), so the candidate blocks of Mirror i
// are mask_i | mask_master. Their number per layer is known before any K/V is read, which
// gives every candidate block a fixed place in the store:
//   prep    per agent: rank of each token in its selection, selection bitmask
//   cand    candidate masks, per-word and per-agent prefix counts, the bound
//           nl * sum_i |cand_i|, master sanity
//   main    one CTA per (layer, 16-token block): reads the canonical tile once, builds
//           the Master's tile (recomputed tokens turned back by R(-off)) and writes it,
//           then for each candidate Mirror builds its tile, compares it bit for bit with
//           the Master's (one block-wide OR) and writes it at its candidate place
//   rows    per (agent, layer) record counts and their prefix sum (rowptr)
//   index   block indices and the (agent, layer, block) -> record slot map
//   fixup   only when some candidate equalled the Master's block: rewrite the kept
//           blocks whose record moved (recomputed from the inputs, never copied)
// No Mirror is built densely; the canonical and recomputed inputs are read once in the
// common case.
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
  const int S = a.rd.S, k = a.k, nbw = a.sc.nbw;
  int32_t* rank = a.sc.rank + static_cast<int64_t>(i) * S;
  const int32_t* sel = a.sel + static_cast<int64_t>(i) * k;
  for (int t = threadIdx.x; t < S; t += blockDim.x) rank[t] = -1;
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) smask[w] = 0u;
  __syncthreads();
  for (int r = threadIdx.x; r < k; r += blockDim.x) {
    const int t = __ldg(sel + r);
    if (t < 0 || t >= S) {
      atomicOr(a.err, err_bit(TD_ERR_INVALID_ARG));
      continue;
    }
    rank[t] = r;
    const int b = t / kDiffBlock;
    atomicOr(&smask[b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  for (int r = threadIdx.x; r < k; r += blockDim.x) {  // duplicates leave a mismatch
    const int t = __ldg(sel + r);
    if (t >= 0 && t < S && rank[t] != r) atomicOr(a.err, err_bit(TD_ERR_INVALID_ARG));
  }
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

// Agent `ag`'s canonical-frame tile items: recomputed K turned back by R(-off) and
// recomputed V at its selected tokens, the canonical K/V elsewhere.
template <int kItems>
__device__ __forceinline__ void agent_tile(const EncArgs& a, int ag, int li,
                                           const int* tok, const int* blk, const int* e0,
                                           const int* f0, const bool* live, const uint4* ka,
                                           const uint4* kb, const uint4* va, const uint4* vb,
                                           uint4* xa, uint4* xb, uint4* ya, uint4* yb) {
  const int S = a.rd.S, E = a.g.E;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    xa[r] = ka[r]; xb[r] = kb[r]; ya[r] = va[r]; yb[r] = vb[r];
    if (!live[r]) continue;
    const int rk = a.sc.rank[static_cast<int64_t>(ag) * S + tok[r]];
    if (rk < 0) continue;
    const int64_t row = ((static_cast<int64_t>(ag) * a.nl + li) * a.k + rk) * E;
    const uint4 fa = ldg16(a.kf + row + e0[r]);
    const uint4 fb = ldg16(a.kf + row + e0[r] + a.g.half);
    const int64_t toff = static_cast<int64_t>(ag * a.rd.M + blk[r]) * a.g.half + f0[r];
    rotate_pairs<true>(fa, fb, a.rd.cos_t + toff, a.rd.sin_t + toff, xa[r], xb[r]);
    ya[r] = ldg16(a.vf + row + e0[r]);
    yb[r] = ldg16(a.vf + row + e0[r] + a.g.half);
  }
}

template <int kItems>
__device__ __forceinline__ void load_canon(const EncArgs& a, int li, int t0, int* tok,
                                           int* blk, int* e0, int* f0, bool* live,
                                           bool* pad, uint4* ka, uint4* kb, uint4* va,
                                           uint4* vb) {
  const int n_items = kDiffBlock * a.g.vpt;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = threadIdx.x + r * blockDim.x;
    const Item it = item_of(a.g, q < n_items ? q : 0);
    tok[r] = t0 + it.tok;
    e0[r] = it.e0;
    f0[r] = it.f0;
    pad[r] = q < n_items && tok[r] >= a.rd.S;    // tail of the last block: zeros
    live[r] = q < n_items && tok[r] < a.rd.S;
    blk[r] = 0;
    ka[r] = kb[r] = va[r] = vb[r] = make_uint4(0u, 0u, 0u, 0u);
    if (live[r]) {
      const int64_t row = (static_cast<int64_t>(li) * a.rd.S + tok[r]) * a.g.E;
      ka[r] = ldg16(a.kc + row + it.e0);
      kb[r] = ldg16(a.kc + row + it.e0 + a.g.half);
      va[r] = ldg16(a.vc + row + it.e0);
      vb[r] = ldg16(a.vc + row + it.e0 + a.g.half);
      blk[r] = __ldg(a.rd.tok_block + tok[r]);
    }
  }
}

template <int kItems>
__device__ __forceinline__ void write_record(const EncArgs& a, int64_t rec, const int* tok,
                                             const int* e0, const bool* live, const bool* pad,
                                             const uint4* xa, const uint4* xb,
                                             const uint4* ya, const uint4* yb, int t0) {
  const int E = a.g.E;
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    if (!live[r] && !pad[r]) continue;
    const int64_t row = (rec * kDiffBlock + (tok[r] - t0)) * E;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    st16(a.store.val_k + row + e0[r], live[r] ? xa[r] : z);
    st16(a.store.val_k + row + e0[r] + a.g.half, live[r] ? xb[r] : z);
    st16(a.store.val_v + row + e0[r], live[r] ? ya[r] : z);
    st16(a.store.val_v + row + e0[r] + a.g.half, live[r] ? yb[r] : z);
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

template <int kItems>
__global__ void __launch_bounds__(256) enc_main_kernel(EncArgs a, int tiles_per_layer) {
  const int m = *a.m_ok;
  if (m < 0) return;
  const int over = *a.over;
  const int tile = blockIdx.x;
  const int li = tile / tiles_per_layer;
  const int b = tile - li * tiles_per_layer;
  const int t0 = b * kDiffBlock;
  const int N = a.rd.N, S = a.rd.S, E = a.g.E, nb = a.rd.nb, nbw = a.sc.nbw;

  int tok[kItems], blk[kItems], e0[kItems], f0[kItems];
  bool live[kItems], pad[kItems];
  uint4 ka[kItems], kb[kItems], va[kItems], vb[kItems];
  load_canon<kItems>(a, li, t0, tok, blk, e0, f0, live, pad, ka, kb, va, vb);

  uint4 mka[kItems], mkb[kItems], mva[kItems], mvb[kItems];
  agent_tile<kItems>(a, m, li, tok, blk, e0, f0, live, ka, kb, va, vb, mka, mkb, mva, mvb);
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    if (!live[r]) continue;
    const int64_t row = (static_cast<int64_t>(li) * S + tok[r]) * E;
    st16(a.store.master_k + row + e0[r], mka[r]);
    st16(a.store.master_k + row + e0[r] + a.g.half, mkb[r]);
    st16(a.store.master_v + row + e0[r], mva[r]);
    st16(a.store.master_v + row + e0[r] + a.g.half, mvb[r]);
  }

  for (int i = 0; i < N; ++i) {
    const unsigned word = a.sc.cand[i * nbw + (b >> 5)];
    const bool is_cand = (word >> (b & 31)) & 1u;
    uint8_t* flag = a.sc.flag + (static_cast<int64_t>(i) * a.nl + li) * nb + b;
    if (!is_cand) {
      if (threadIdx.x == 0) *flag = 0;
      continue;
    }
    uint4 xa[kItems], xb[kItems], ya[kItems], yb[kItems];
    agent_tile<kItems>(a, i, li, tok, blk, e0, f0, live, ka, kb, va, vb, xa, xb, ya, yb);
    bool d = false;
#pragma unroll
    for (int r = 0; r < kItems; ++r)
      if (live[r])
        d |= neq16(xa[r], mka[r]) | neq16(xb[r], mkb[r]) | neq16(ya[r], mva[r]) |
             neq16(yb[r], mvb[r]);
    const int differs = __syncthreads_or(d);
    if (threadIdx.x == 0) *flag = differs ? 1 : 0;
    if (!over && differs)
      write_record<kItems>(a, cand_place(a, i, li, b), tok, e0, live, pad, xa, xb, ya, yb, t0);
  }
}

// Record counts per (agent, layer) row and their exclusive prefix sum.
__global__ void __launch_bounds__(1024) enc_rows_kernel(EncArgs a) {
  extern __shared__ long long rcnt[];  // [R]
  __shared__ long long wsum[32];
  if (*a.m_ok < 0) return;
  const int R = a.rd.N * a.nl, nb = a.rd.nb;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int r = wid; r < R; r += nw) {
    const uint8_t* f = a.sc.flag + static_cast<int64_t>(r) * nb;
    int c = 0;
    for (int b = lane; b < nb; b += 32) c += f[b];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) rcnt[r] = c;
  }
  __syncthreads();
  // exclusive scan over R rows: each thread a contiguous chunk
  const int per = (R + blockDim.x - 1) / blockDim.x;
  const int r0 = threadIdx.x * per, r1 = min(R, r0 + per);
  long long local = 0;
  for (int r = r0; r < r1; ++r) local += rcnt[r];
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
    const long long c = rcnt[r];
    a.store.rowptr[r] = run;
    run += c;
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
  const uint8_t* f = a.sc.flag + w * nb;
  int32_t* slot = a.store.slot + w * nb;
  int64_t run = a.store.rowptr[w];
  for (int b0 = 0; b0 < nb; b0 += 32) {
    const int b = b0 + lane;
    const bool on = b < nb && f[b];
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, on);
    const int64_t pos = run + __popc(bal & ((1u << lane) - 1u));
    if (b < nb) slot[b] = on ? static_cast<int32_t>(pos) : -1;
    if (on) a.store.block_idx[pos] = b;
    run += __popc(bal);
  }
}

// Rewrites the kept blocks whose record is not at their candidate place (only when some
// candidate turned out equal to the Master's block).
template <int kItems>
__global__ void __launch_bounds__(256) enc_fixup_kernel(EncArgs a, int tiles_per_layer) {
  if (*a.sc.need_fixup == 0) return;
  const int m = *a.m_ok;
  if (m < 0) return;
  const int tile = blockIdx.x;
  const int li = tile / tiles_per_layer;
  const int b = tile - li * tiles_per_layer;
  const int t0 = b * kDiffBlock;
  int tok[kItems], blk[kItems], e0[kItems], f0[kItems];
  bool live[kItems], pad[kItems];
  uint4 ka[kItems], kb[kItems], va[kItems], vb[kItems];
  load_canon<kItems>(a, li, t0, tok, blk, e0, f0, live, pad, ka, kb, va, vb);
  for (int i = 0; i < a.rd.N; ++i) {
    if (i == m) continue;
    const int s = a.store.slot[(static_cast<int64_t>(i) * a.nl + li) * a.rd.nb + b];
    if (s < 0 || s == cand_place(a, i, li, b)) continue;
    uint4 xa[kItems], xb[kItems], ya[kItems], yb[kItems];
    agent_tile<kItems>(a, i, li, tok, blk, e0, f0, live, ka, kb, va, vb, xa, xb, ya, yb);
    write_record<kItems>(a, s, tok, e0, live, pad, xa, xb, ya, yb, t0);
  }
}

template <int kItems>
static cudaError_t run_tiles(const EncArgs& a, int threads, cudaStream_t st) {
  const int tpl = a.rd.nb;
  const int64_t tiles = static_cast<int64_t>(tpl) * a.nl;
  enc_main_kernel<kItems><<<static_cast<unsigned>(tiles), threads, 0, st>>>(a, tpl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t rows_smem = static_cast<size_t>(a.rd.N) * a.nl * sizeof(long long);
  if (rows_smem > 48 * 1024) {
    e = cudaFuncSetAttribute(enc_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(rows_smem));
    if (e != cudaSuccess) return e;
  }
  enc_rows_kernel<<<1, 1024, rows_smem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.rd.N) * a.nl;
  enc_index_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  enc_fixup_kernel<kItems><<<static_cast<unsigned>(tiles), threads, 0, st>>>(a, tpl);
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
  enc_prep_kernel<<<rd.N, 1024, sc.nbw * sizeof(unsigned), st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  enc_cand_kernel<<<1, 1024, 0, st>>>(a, master);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int threads = tile_threads(g);
  const int per = (kDiffBlock * g.vpt + threads - 1) / threads;
  if (per <= 1) return run_tiles<1>(a, threads, st);
  if (per <= 2) return run_tiles<2>(a, threads, st);
  if (per <= 4) return run_tiles<4>(a, threads, st);
  return run_tiles<8>(a, threads, st);
}

}  // namespace td
