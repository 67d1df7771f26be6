// k_restore.cu - stage 4: fused diff restore (TokenDance review [R], Summary Method (3): on
// read-back, merge each Mirror's diffs into the Master's data in flight and recover RoPE,
// without building a dense Mirror; §2a "Fused restore: Master chunk + diff -> paged KV";
// §3d: recovery belongs in the transfer path, written through the paged-KV slot map).
//
// One CTA per unit = (layer, one 16-token tile, K or V, part). The Master's data of the
// unit is read from HBM once and held in registers; for each listed agent the slot map
// says whether that agent has a record for the tile's diff block (16 or 32 tokens) in
// this layer: if so the record's rows replace the Master's data for this agent only. K is turned by the agent's block
// offsets (frame 0) or copied (frame 1), V is copied; 16-byte stores into the agent's
// page.
#include "td_device.cuh"

namespace td {

template <int kItems, bool kRotate>
__global__ void __launch_bounds__(256, 3)
restore_kernel(Geom g, RoundDev rd, PoolDev pool, StoreDev store, AgentList agents,
               int layer_begin, int store_layer0, int tiles_per_layer, uint32_t* err) {
  pdl_wait();
  __shared__ int64_t s_row[kAgentChunk * kTile];  // pool row of (agent, token)
  __shared__ int s_rec[kAgentChunk];               // record of (agent), -1 none, -2 bad
  const Unit un = unit_of(g, blockIdx.x, tiles_per_layer);
  const int t0 = un.b * kTile;
  const int db = t0 / rd.B;                        // the tile's diff block
  const int tb0 = t0 - db * rd.B;                  // the tile's first row within it
  const int layer = layer_begin + un.li;
  const int sl = layer - store_layer0;              // layer index within the store
  const int n_items = kTile * g.vpt;
  const uint16_t* master = un.kv == 0 ? store.master_k : store.master_v;
  const uint16_t* vals = un.kv == 0 ? store.val_k : store.val_v;

  uint4 ma[kItems], mb[kItems];
  int e0[kItems], f0[kItems], tl[kItems], blk[kItems];
  bool live[kItems];
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = un.q0 + threadIdx.x + r * blockDim.x;
    const Item it = item_of(g, q < n_items ? q : 0);
    const int t = t0 + it.tok;
    live[r] = q < n_items && t < rd.S;
    e0[r] = it.e0;
    f0[r] = it.f0;
    tl[r] = it.tok;
    blk[r] = 0;
    if (live[r]) {
      const int64_t row = (static_cast<int64_t>(sl) * rd.S + t) * g.E;
      ma[r] = ldg16(master + row + it.e0);
      mb[r] = ldg16(master + row + it.e0 + g.half);
      blk[r] = __ldg(rd.tok_block + t);
    }
  }

  for (int c0 = 0; c0 < agents.n; c0 += kAgentChunk) {
    const int n = min(kAgentChunk, agents.n - c0);
    if (c0 > 0) __syncthreads();  // the previous chunk's tables are no longer read
    chunk_rows(rd, pool, layer, un.kv, t0, n, [&](int x) { return agents.a[c0 + x]; }, s_row,
               err);
    for (int x = threadIdx.x; x < n; x += blockDim.x) {
      const int a = agents.a[c0 + x];
      int rec = __ldg(store.slot + (static_cast<int64_t>(a) * store.nl + sl) * rd.nb + db);
      if (rec >= store.capacity) {  // a slot map that does not belong to this store
        atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
        rec = -2;
      }
      s_rec[x] = rec;
    }
    __syncthreads();

    // source of agent x: its record, or the Master; fetched one agent ahead
    uint4 na[kItems], nb[kItems];
    auto fetch = [&](int x) {
      const int rec = s_rec[x];
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        na[r] = ma[r];
        nb[r] = mb[r];
        if (live[r] && rec >= 0) {
          const int64_t row = (static_cast<int64_t>(rec) * rd.B + tb0 + tl[r]) * g.E;
          na[r] = ldg16(vals + row + e0[r]);
          nb[r] = ldg16(vals + row + e0[r] + g.half);
        }
      }
    };
    fetch(0);
    for (int x = 0; x < n; ++x) {
      uint4 ca[kItems], cb[kItems];
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        ca[r] = na[r];
        cb[r] = nb[r];
      }
      const bool skip = s_rec[x] == -2;
      if (x + 1 < n) fetch(x + 1);
      if (skip) continue;
      const int a = agents.a[c0 + x];
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (!live[r]) continue;
        const int64_t row = s_row[x * kTile + tl[r]];
        if (row < 0) continue;
        uint16_t* dst = pool.base + row * g.E;
        uint4 sa = ca[r], sb = cb[r];
        if (kRotate && un.kv == 0) {
          const int64_t toff = static_cast<int64_t>(a * rd.M + blk[r]) * g.half + f0[r];
          rotate_pairs<false>(ca[r], cb[r], rd.cos_t + toff, rd.sin_t + toff, sa, sb);
        }
        st16(dst + e0[r], sa);
        st16(dst + e0[r] + g.half, sb);
      }
    }
  }
}

template <int kItems>
static cudaError_t go(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                      const StoreDev& store, const AgentList& agents, int layer_begin,
                      int store_layer0, int nl, int frame, uint32_t* err, cudaStream_t st) {
  const int tpl = rd.nt;
  const int64_t units = static_cast<int64_t>(tpl) * nl * 2 * parts_per_tile(g);
  if (units == 0 || agents.n == 0) return cudaSuccess;
  if (frame == 0)
    return launch_after(restore_kernel<kItems, true>, static_cast<unsigned>(units),
                        tile_threads(g), 0, st, g, rd, pool, store, agents, layer_begin,
                        store_layer0, tpl, err);
  return launch_after(restore_kernel<kItems, false>, static_cast<unsigned>(units),
                      tile_threads(g), 0, st, g, rd, pool, store, agents, layer_begin,
                      store_layer0, tpl, err);
}

cudaError_t launch_restore(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                           const StoreDev& store, const AgentList& agents, int layer_begin,
                           int store_layer0, int nl, int frame, uint32_t* err,
                           cudaStream_t st) {
  if (tile_items(g) == 1)
    return go<1>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
  return go<2>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
}

// The dense restore the fused restore replaces ([R] §3d; Figure 5's "dense Mirror"): one
// agent's canonical-frame cache materialised as [layer][token][E] K and V, the Master's
// rows with the agent's records laid over them. One CTA per (layer, diff block, K or V)
// copies the block's rows with 16-byte loads and stores. A comparison baseline only.
__global__ void __launch_bounds__(256)
materialise_kernel(int E, int S, int B, int nb, StoreDev store, int agent, int sl0,
                   uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, uint32_t* err) {
  pdl_wait();
  const int kv = blockIdx.x & 1;
  const int b = (blockIdx.x >> 1) % nb;
  const int li = (blockIdx.x >> 1) / nb;
  const int sl = sl0 + li;
  int rec = __ldg(store.slot + (static_cast<int64_t>(agent) * store.nl + sl) * nb + b);
  if (rec >= store.capacity) {
    if (threadIdx.x == 0) atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
    return;
  }
  const int t0 = b * B;
  const int ntok = min(B, S - t0);
  const int vpt = E / 8;
  const uint16_t* src = rec >= 0
      ? (kv ? store.val_v : store.val_k) + static_cast<int64_t>(rec) * B * E
      : (kv ? store.master_v : store.master_k) + (static_cast<int64_t>(sl) * S + t0) * E;
  uint16_t* dst = (kv ? dv : dk) + (static_cast<int64_t>(li) * S + t0) * E;
  for (int v = threadIdx.x; v < ntok * vpt; v += blockDim.x)
    st16(dst + static_cast<int64_t>(v) * 8, ldg16(src + static_cast<int64_t>(v) * 8));
}

cudaError_t launch_materialise(const Geom& g, const RoundDev& rd, const StoreDev& store,
                               int agent, int sl0, int nl, uint16_t* dk, uint16_t* dv,
                               uint32_t* err, cudaStream_t st) {
  const int64_t units = static_cast<int64_t>(nl) * rd.nb * 2;
  if (units == 0) return cudaSuccess;
  return launch_after(materialise_kernel, static_cast<unsigned>(units), 256, 0, st, g.E, rd.S,
                      rd.B, rd.nb, store, agent, sl0, dk, dv, err);
}

}  // namespace td
