// k_rerotate.cu - stage 1: collective re-rotation of the shared blocks into every agent's
// paged KV (TokenDance review [R], Summary Method (2) and Figure 7 T3: one RoPE pass for
// the whole group of agents instead of one per request).
//
// One CTA per unit = (layer, 16 canonical tokens, K or V, part of at most 512 pair-
// vectors). The unit's canonical data is read from HBM once, kept in registers and written
// N times: for each agent a K unit turns its pair-vectors by that agent's block-offset
// angles, a V unit copies; every thread stores 16-byte vectors into the agent's page.
// HBM traffic per tile: 16*E*2 bytes read per tensor, N times that written.
#include "td_device.cuh"

namespace td {

template <int kItems>
__global__ void __launch_bounds__(256, 4)
rerotate_kernel(Geom g, RoundDev rd, PoolDev pool, const uint16_t* __restrict__ kc,
                const uint16_t* __restrict__ vc, int layer_begin, int tiles_per_layer,
                uint32_t* err) {
  pdl_wait();
  __shared__ int64_t s_row[kAgentChunk * kTile];  // pool row of (agent, token)
  const Unit un = unit_of(g, blockIdx.x, tiles_per_layer);
  if (un.kv == 1 && vc == nullptr) return;
  const uint16_t* src = un.kv == 0 ? kc : vc;
  const int t0 = un.b * kTile;
  const int layer = layer_begin + un.li;
  const int n_items = kTile * g.vpt;

  uint4 xa[kItems], xb[kItems];
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
      const uint16_t* row = src + (static_cast<int64_t>(un.li) * rd.S + t) * g.E;
      xa[r] = ldg16(row + it.e0);
      xb[r] = ldg16(row + it.e0 + g.half);
      blk[r] = __ldg(rd.tok_block + t);
    }
  }

  for (int c0 = 0; c0 < rd.N; c0 += kAgentChunk) {
    const int n = min(kAgentChunk, rd.N - c0);
    if (c0 > 0) __syncthreads();  // the previous chunk's rows are no longer read
    chunk_rows(rd, pool, layer, un.kv, t0, n, [&](int x) { return c0 + x; }, s_row, err);
    __syncthreads();
    for (int x = 0; x < n; ++x) {
      const int i = c0 + x;
#pragma unroll
      for (int r = 0; r < kItems; ++r) {
        if (!live[r]) continue;
        const int64_t row = s_row[x * kTile + tl[r]];
        if (row < 0) continue;
        uint16_t* dst = pool.base + row * g.E;
        if (un.kv == 0) {
          const int64_t toff = static_cast<int64_t>(i * rd.M + blk[r]) * g.half + f0[r];
          uint4 ya, yb;
          rotate_pairs<false>(xa[r], xb[r], rd.cos_t + toff, rd.sin_t + toff, ya, yb);
          st16(dst + e0[r], ya);
          st16(dst + e0[r] + g.half, yb);
        } else {
          st16(dst + e0[r], xa[r]);
          st16(dst + e0[r] + g.half, xb[r]);
        }
      }
    }
  }
}

int tile_threads(const Geom& g) {
  const int items = kTile * g.vpt < kPartItems ? kTile * g.vpt : kPartItems;
  return items < 256 ? items : 256;
}

int tile_items(const Geom& g) {
  const int items = kTile * g.vpt < kPartItems ? kTile * g.vpt : kPartItems;
  const int t = tile_threads(g);
  return (items + t - 1) / t;
}

cudaError_t launch_rerotate(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                            const uint16_t* kc, const uint16_t* vc, int layer_begin, int nl,
                            uint32_t* err, cudaStream_t st) {
  const int tpl = (rd.S + kTile - 1) / kTile;
  const int64_t units = static_cast<int64_t>(tpl) * nl * 2 * parts_per_tile(g);
  if (units == 0) return cudaSuccess;
  if (tile_items(g) == 1)
    return launch_after(rerotate_kernel<1>, static_cast<unsigned>(units), tile_threads(g), 0, st,
                        g, rd, pool, kc, vc, layer_begin, tpl, err);
  return launch_after(rerotate_kernel<2>, static_cast<unsigned>(units), tile_threads(g), 0, st,
                      g, rd, pool, kc, vc, layer_begin, tpl, err);
}

}  // namespace td
