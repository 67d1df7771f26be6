// k_restore.cu - stage 4: fused diff restore (TokenDance review [R], Summary Method (3): on
// read-back, merge each Mirror's diffs into the Master's data in flight and recover RoPE,
// without building a dense Mirror; §2a "Fused restore: Master chunk + diff -> paged KV";
// §3d: recovery belongs in the transfer path, written through the paged-KV slot map).
//
// One CTA per tile = (layer, one 16-token diff block). The Master's tile is read from HBM
// once and held in registers; for each listed agent the slot map says whether that agent
// has a record for this (layer, block): if so its record replaces the Master's tile for
// this agent only. K is turned by the agent's block offsets (frame 0) or copied (frame 1),
// V is copied, both stored 16 bytes per thread into the agent's page.
#include "td_device.cuh"

namespace td {

template <int kItems, bool kRotate>
__global__ void __launch_bounds__(256)
restore_kernel(Geom g, RoundDev rd, PoolDev pool, StoreDev store, AgentList agents,
               int layer_begin, int store_layer0, int tiles_per_layer, uint32_t* err) {
  const int tile = blockIdx.x;
  const int li = tile / tiles_per_layer;            // layer index within this call
  const int b = tile - li * tiles_per_layer;
  const int t0 = b * kDiffBlock;
  const int layer = layer_begin + li;
  const int sl = layer - store_layer0;              // layer index within the store
  const int n_items = kDiffBlock * g.vpt;

  uint4 ka[kItems], kb[kItems], va[kItems], vb[kItems];
  int e0[kItems], f0[kItems], tl[kItems], blk[kItems], u[kItems];
  bool live[kItems];
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = threadIdx.x + r * blockDim.x;
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
      ka[r] = ldg16(store.master_k + row + it.e0);
      kb[r] = ldg16(store.master_k + row + it.e0 + g.half);
      va[r] = ldg16(store.master_v + row + it.e0);
      vb[r] = ldg16(store.master_v + row + it.e0 + g.half);
      blk[r] = __ldg(rd.tok_block + t);
      u[r] = t - __ldg(rd.blk_start + blk[r]);
    }
  }

  for (int x = 0; x < agents.n; ++x) {
    const int a = agents.a[x];
    int rec = __ldg(store.slot + (static_cast<int64_t>(a) * store.nl + sl) * rd.nb + b);
    if (rec >= store.capacity) {  // a slot map that does not belong to this store
      if (threadIdx.x == 0) atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
      continue;
    }
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
      if (!live[r]) continue;
      uint4 sa = ka[r], sb = kb[r], wa = va[r], wb = vb[r];
      if (rec >= 0) {
        const int64_t row = (static_cast<int64_t>(rec) * kDiffBlock + tl[r]) * g.E;
        sa = ldg16(store.val_k + row + e0[r]);
        sb = ldg16(store.val_k + row + e0[r] + g.half);
        wa = ldg16(store.val_v + row + e0[r]);
        wb = ldg16(store.val_v + row + e0[r] + g.half);
      }
      const int ab = a * rd.M + blk[r];
      const int pos = __ldg(rd.off + ab) + u[r];
      uint16_t* kdst = pool_row(pool, g.E, a, layer, 0, pos, err);
      if (!kdst) continue;
      if (kRotate) {
        const int64_t toff = static_cast<int64_t>(ab) * g.half + f0[r];
        uint4 ya, yb;
        rotate_pairs<false>(sa, sb, rd.cos_t + toff, rd.sin_t + toff, ya, yb);
        sa = ya;
        sb = yb;
      }
      st16(kdst + e0[r], sa);
      st16(kdst + e0[r] + g.half, sb);
      uint16_t* vdst = kdst + pool.num_pages * static_cast<int64_t>(pool.P) * g.E;
      st16(vdst + e0[r], wa);
      st16(vdst + e0[r] + g.half, wb);
    }
  }
}

template <int kItems>
static cudaError_t go(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                      const StoreDev& store, const AgentList& agents, int layer_begin,
                      int store_layer0, int nl, int frame, uint32_t* err, cudaStream_t st) {
  const int tpl = rd.nb;
  const int64_t tiles = static_cast<int64_t>(tpl) * nl;
  if (tiles == 0 || agents.n == 0) return cudaSuccess;
  if (frame == 0)
    restore_kernel<kItems, true><<<static_cast<unsigned>(tiles), tile_threads(g), 0, st>>>(
        g, rd, pool, store, agents, layer_begin, store_layer0, tpl, err);
  else
    restore_kernel<kItems, false><<<static_cast<unsigned>(tiles), tile_threads(g), 0, st>>>(
        g, rd, pool, store, agents, layer_begin, store_layer0, tpl, err);
  return cudaGetLastError();
}

cudaError_t launch_restore(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                           const StoreDev& store, const AgentList& agents, int layer_begin,
                           int store_layer0, int nl, int frame, uint32_t* err,
                           cudaStream_t st) {
  const int items = kDiffBlock * g.vpt;
  const int per = (items + tile_threads(g) - 1) / tile_threads(g);
  if (per <= 1) return go<1>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
  if (per <= 2) return go<2>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
  if (per <= 4) return go<4>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
  return go<8>(g, rd, pool, store, agents, layer_begin, store_layer0, nl, frame, err, st);
}

}  // namespace td
