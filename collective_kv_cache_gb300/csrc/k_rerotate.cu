// k_rerotate.cu - stage 1: collective re-rotation of the shared blocks into every agent's
// paged KV (TokenDance review [R], Summary Method (2) and Figure 7 T3: one RoPE pass for
// the whole group of agents instead of one per request).
//
// One CTA per tile = (layer, 16 canonical tokens). The tile's canonical K/V are read from
// HBM once, kept in registers, and written N times: for each agent the K pair-vectors are
// turned by that agent's (block offset) angles and both K and V are stored, 16 bytes per
// thread per vector, into the agent's page. HBM traffic per tile: 16*E*2 bytes read per
// tensor, N times that written.
#include "td_device.cuh"

namespace td {

template <int kItems>
__global__ void __launch_bounds__(256)
rerotate_kernel(Geom g, RoundDev rd, PoolDev pool, const uint16_t* __restrict__ kc,
                const uint16_t* __restrict__ vc, int layer_begin, int tiles_per_layer,
                uint32_t* err) {
  const int tile = blockIdx.x;
  const int li = tile / tiles_per_layer;
  const int t0 = (tile - li * tiles_per_layer) * kDiffBlock;
  const int layer = layer_begin + li;
  const int n_items = kDiffBlock * g.vpt;

  uint4 ka[kItems], kb[kItems], va[kItems], vb[kItems];
  int e0[kItems], f0[kItems], tok[kItems], blk[kItems], u[kItems];
  bool live[kItems];
#pragma unroll
  for (int r = 0; r < kItems; ++r) {
    const int q = threadIdx.x + r * blockDim.x;
    const Item it = item_of(g, q < n_items ? q : 0);
    const int t = t0 + it.tok;
    live[r] = q < n_items && t < rd.S;
    e0[r] = it.e0;
    f0[r] = it.f0;
    tok[r] = t;
    blk[r] = 0;
    u[r] = 0;
    if (live[r]) {
      const uint16_t* row = kc + (static_cast<int64_t>(li) * rd.S + t) * g.E;
      ka[r] = ldg16(row + it.e0);
      kb[r] = ldg16(row + it.e0 + g.half);
      if (vc) {
        const uint16_t* vrow = vc + (static_cast<int64_t>(li) * rd.S + t) * g.E;
        va[r] = ldg16(vrow + it.e0);
        vb[r] = ldg16(vrow + it.e0 + g.half);
      }
      blk[r] = __ldg(rd.tok_block + t);
      u[r] = t - __ldg(rd.blk_start + blk[r]);
    }
  }

  for (int i = 0; i < rd.N; ++i) {
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
      if (!live[r]) continue;
      const int ab = i * rd.M + blk[r];
      const int pos = __ldg(rd.off + ab) + u[r];
      uint16_t* kdst = pool_row(pool, g.E, i, layer, 0, pos, err);
      if (!kdst) continue;
      const int64_t toff = static_cast<int64_t>(ab) * g.half + f0[r];
      uint4 ya, yb;
      rotate_pairs<false>(ka[r], kb[r], rd.cos_t + toff, rd.sin_t + toff, ya, yb);
      st16(kdst + e0[r], ya);
      st16(kdst + e0[r] + g.half, yb);
      if (vc) {
        uint16_t* vdst = kdst + pool.num_pages * static_cast<int64_t>(pool.P) * g.E;
        st16(vdst + e0[r], va[r]);
        st16(vdst + e0[r] + g.half, vb[r]);
      }
    }
  }
  (void)tok;
}

int tile_threads(const Geom& g) {
  const int items = kDiffBlock * g.vpt;
  return items < 256 ? items : 256;
}

template <int kItems>
static cudaError_t go(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                      const uint16_t* kc, const uint16_t* vc, int layer_begin, int nl,
                      uint32_t* err, cudaStream_t st) {
  const int tiles_per_layer = (rd.S + kDiffBlock - 1) / kDiffBlock;
  const int64_t tiles = static_cast<int64_t>(tiles_per_layer) * nl;
  if (tiles == 0) return cudaSuccess;
  rerotate_kernel<kItems><<<static_cast<unsigned>(tiles), tile_threads(g), 0, st>>>(
      g, rd, pool, kc, vc, layer_begin, tiles_per_layer, err);
  return cudaGetLastError();
}

cudaError_t launch_rerotate(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                            const uint16_t* kc, const uint16_t* vc, int layer_begin, int nl,
                            uint32_t* err, cudaStream_t st) {
  const int items = kDiffBlock * g.vpt;
  const int per = (items + tile_threads(g) - 1) / tile_threads(g);
  if (per <= 1) return go<1>(g, rd, pool, kc, vc, layer_begin, nl, err, st);
  if (per <= 2) return go<2>(g, rd, pool, kc, vc, layer_begin, nl, err, st);
  if (per <= 4) return go<4>(g, rd, pool, kc, vc, layer_begin, nl, err, st);
  return go<8>(g, rd, pool, kc, vc, layer_begin, nl, err, st);
}

}  // namespace td
