// k_restore.cu - stage 4: fused diff restore (TokenDance review [R], Summary Method (3): on
// read-back, merge each Mirror's diffs into the Master's data in flight and recover RoPE,
// without building a dense Mirror; §2a "Fused restore: Master chunk + diff -> paged KV";
// §3d: recovery belongs in the transfer path, written through the paged-KV slot map).
//
// One CTA per unit = (layer, one 16-token diff block, K or V, part). The Master's data of
// the unit is read from HBM once and held in registers; for each listed agent the slot
// map says whether that agent has a record for this (layer, block): if so its record
// replaces the Master's data for this agent only. K is turned by the agent's block
// offsets (frame 0) or copied (frame 1), V is copied; 16-byte stores into the agent's
// page.
#include "td_device.cuh"

namespace td {

template <int kItems, bool kRotate>
__global__ void __launch_bounds__(256, 3)
restore_kernel(Geom g, RoundDev rd, PoolDev pool, StoreDev store, AgentList agents,
               int layer_begin, int store_layer0, int tiles_per_layer, uint32_t* err) {
  const Unit un = unit_of(g, blockIdx.x, tiles_per_layer);
  const int t0 = un.b * kDiffBlock;
  const int layer = layer_begin + un.li;
  const int sl = layer - store_layer0;              // layer index within the store
  const int n_items = kDiffBlock * g.vpt;
  const uint16_t* master = un.kv == 0 ? store.master_k : store.master_v;
  const uint16_t* vals = un.kv == 0 ? store.val_k : store.val_v;

  uint4 ma[kItems], mb[kItems];
  int e0[kItems], f0[kItems], tl[kItems], blk[kItems], u[kItems];
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
    u[r] = 0;
    if (live[r]) {
      const int64_t row = (static_cast<int64_t>(sl) * rd.S + t) * g.E;
      ma[r] = ldg16(master + row + it.e0);
      mb[r] = ldg16(master + row + it.e0 + g.half);
      blk[r] = __ldg(rd.tok_block + t);
      u[r] = t - __ldg(rd.blk_start + blk[r]);
    }
  }

  for (int x = 0; x < agents.n; ++x) {
    const int a = agents.a[x];
    const int rec = __ldg(store.slot + (static_cast<int64_t>(a) * store.nl + sl) * rd.nb + un.b);
    if (rec >= store.capacity) {  // a slot map that does not belong to this store
      if (threadIdx.x == 0) atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
      continue;
    }
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
      if (!live[r]) continue;
      uint4 sa = ma[r], sb = mb[r];
      if (rec >= 0) {
        const int64_t row = (static_cast<int64_t>(rec) * kDiffBlock + tl[r]) * g.E;
        sa = ldg16(vals + row + e0[r]);
        sb = ldg16(vals + row + e0[r] + g.half);
      }
      const int ab = a * rd.M + blk[r];
      const int pos = __ldg(rd.off + ab) + u[r];
      uint16_t* dst = pool_row(pool, g.E, a, layer, un.kv, pos, err);
      if (!dst) continue;
      if (kRotate && un.kv == 0) {
        const int64_t toff = static_cast<int64_t>(ab) * g.half + f0[r];
        uint4 ya, yb;
        rotate_pairs<false>(sa, sb, rd.cos_t + toff, rd.sin_t + toff, ya, yb);
        sa = ya;
        sb = yb;
      }
      st16(dst + e0[r], sa);
      st16(dst + e0[r] + g.half, sb);
    }
  }
}

template <int kItems>
static cudaError_t go(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                      const StoreDev& store, const AgentList& agents, int layer_begin,
                      int store_layer0, int nl, int frame, uint32_t* err, cudaStream_t st) {
  const int tpl = rd.nb;
  const int64_t units = static_cast<int64_t>(tpl) * nl * 2 * parts_per_tile(g);
  if (units == 0 || agents.n == 0) return cudaSuccess;
  if (frame == 0)
    restore_kernel<kItems, true><<<static_cast<unsigned>(units), tile_threads(g), 0, st>>>(
        g, rd, pool, store, agents, layer_begin, store_layer0, tpl, err);
  else
    restore_kernel<kItems, false><<<static_cast<unsigned>(units), tile_threads(g), 0, st>>>(
        g, rd, pool, store, agents, layer_begin, store_layer0, tpl, err);
  return cudaGetLastError();
}

cudaError_t launch_restore(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                           const StoreDev& store, const AgentList& agents, int layer_begin,
                           int store_layer0, int nl, int frame, uint32_t* err,
                           cudaStream_t st) {
  if (tile_items(g) == 1)
    return go<1>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
  return go<2>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
}

}  // namespace td
