// k_attention.cu - decode attention read straight from the Master and the diffs (TokenDance
// blog post [B] §4.4 "Fused Diff Restore": the diff is applied block by block on chip and
// attention runs right after, with no materialised cache; review [R] §8, open questions,
// and §9: a paired block-sparse KV diff kernel aligned with FlashAttention).
//
// Agent a's context is its private history, positions [0, h_a) whose K/V its pages hold as
// stored, followed by the shared tokens: the Master's rows with a's records laid over them,
// in the canonical frame. The shared token of block j at local index u sits at position
// off_aj + u with K = R(off_aj) X; instead of turning every key the kernel turns the query
// once per block, q . R(off) X = (R(-off) q) . X, so shared rows are used as stored.
//
// Work unit = (layer, kv head, agent, 512 positions of the agent's context; 128 in the last
// layers), one warp:
//   - the rows of the head (D bf16 per position) are staged in shared memory by the TMA
//     engine from 2-D tensor maps of the pool, the records and the Master (16 x 64 boxes,
//     128-byte swizzle): a stage is at most 16 positions from one page, one diff block and
//     one shared block, so it arrives as D/64 boxes of K and D/64 of V. Two stages ring on
//     mbarriers, 16 KB a warp, so thirteen warps fit on an SM. Every
//     wait is bounded in time (0.2 s by the global timer); on time-out the unit records
//     TD_ERR_DEVICE_TIMEOUT, waits (bounded again) for the copies it issued and returns;
//   - both products on the tensor cores, mma.sync m16n8k16 bf16 with float32 accumulators,
//     the head group's G <= 8 query heads as rows (rows G..15 zero). A turned query is
//     float32: it is split into a bf16 high part and a bf16 low part, two products per
//     k-chunk, so each score keeps 16 bits of the query (a history query is bf16 already:
//     one product); the softmax weights are split the same way for P V;
//   - online softmax in base 2; each lane keeps the statistics of its fragment row (query
//     head), so rescaling needs no exchange;
//   - the next stage's source rows are looked up before this stage's products, so the
//     lookups' latency hides behind them;
//   - the unit writes its partial (max, sum, unnormalised output) of the G query heads;
//     attn_combine_kernel merges an agent's units;
//   - the grid ends with the last layers cut into 128-position units, so that the last
//     units to start are short and the SMs stay busy until close to the end (in 512-position
//     units the final wave left half the SMs idle for the last ~40 us).
// The same kernel with every position read from the pages (kFromPool) is plain paged
// decode attention over a restored cache: the baseline the fusion replaces.
#include "td_device.cuh"

namespace td {

namespace {

// One box of a 2-D tensor map (16 rows x 64 bf16, 128-byte swizzle) into shared memory;
// x = column (elements), y = row; completion counted on `bar`.
__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int x, int y,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled box (rows of 128 bytes,
// chunk c stored at c ^ (r mod 8); the box starts on a 1024-byte boundary).
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D += A * B, m16n8k16, bf16 inputs, float32 accumulators, all four A registers given.
__device__ __forceinline__ void mma_bf16_full(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return static_cast<uint16_t>(pack_bf2(x, 0.0f) & 0xFFFFu);
}

}  // namespace

template <int D, bool kFromPool>
__global__ void __launch_bounds__(32, 13)
attn_unit_kernel(const __grid_constant__ AttnArgs A, const __grid_constant__ AttnList list,
                 const __grid_constant__ AttnMaps maps) {
  pdl_wait();
  constexpr int KCH = D / 16;         // k-chunks of one q.k product
  constexpr int HALVES = D / 64;      // 64-column boxes per row (a box row is 128 bytes)
  constexpr int BOX = kAttnStage * 128;               // one box: 16 rows x 128 bytes
  constexpr int TILE = HALVES * BOX;                  // one stage of K (or V)
  __shared__ __align__(1024) unsigned char s_k[kAttnDepth][TILE];
  __shared__ __align__(1024) unsigned char s_v[kAttnDepth][TILE];
  __shared__ __align__(8) uint64_t s_bar[kAttnDepth];

  const int lane = threadIdx.x;
  const int gid = lane >> 2, tig = lane & 3;   // mma fragment group / thread in group
  // the unit: layers [0, split) in long units first, then the rest in short ones
  const int64_t n_long = static_cast<int64_t>(list.split) * A.g.H * list.base[list.n];
  const bool short_unit = static_cast<int64_t>(blockIdx.x) >= n_long;
  const int32_t* base = short_unit ? list.base2 : list.base;
  const int ch = short_unit ? kAttnTailChunk : kAttnChunk;
  const int total = base[list.n];
  int64_t u = short_unit ? blockIdx.x - n_long : blockIdx.x;
  const int c = static_cast<int>(u % total);
  u /= total;
  const int h = static_cast<int>(u % A.g.H);
  const int li = static_cast<int>(u / A.g.H) + (short_unit ? list.split : 0);
  int lo = 0, hi = list.n - 1;                 // the agent of unit c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  const int x = lo, a = list.a[x];
  const int S = A.rd.S, P = A.pool.P;
  const int n_ctx = list.hist[x] + S;
  const int hist = kFromPool ? n_ctx : list.hist[x];   // positions read from the pages
  // units of an agent: its history in chunks of ch positions, then its shared tokens in
  // chunks of ch tokens (so no unit straddles the two and every stage starts aligned)
  const int nh = (hist + ch - 1) / ch;
  const int cu = c - base[x];
  const int p0 = cu < nh ? cu * ch : hist + (cu - nh) * ch;
  const int p1 = cu < nh ? min(p0 + ch, hist) : min(p0 + ch, n_ctx);
  const int layer = A.layer_begin + li, sl = A.sl0 + li;

  if (lane < kAttnDepth) mbar_init(&s_bar[lane], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();

  // the stage that starts at position p: at most 16 positions from one place, so one box
  // holds them: within a page (history), or within a shared block and a diff block
  auto stage_end = [&](int p) {
    int e;
    if (p < hist) {
      e = min((p / P + 1) * P, hist);
    } else {
      const int t = p - hist;
      const int j = __ldg(A.rd.tok_block + t);
      const int blk_end = j + 1 < A.rd.M ? __ldg(A.rd.blk_start + j + 1) : S;
      e = hist + min(blk_end, (t / A.rd.B + 1) * A.rd.B);
    }
    return min(min(p + kAttnStage, e), p1);
  };
  auto segment = [&](int p) { return p < hist ? -1 : __ldg(A.rd.tok_block + (p - hist)); };

  // lane 0 fires the stage at p: K and V boxes (HALVES each) from the page, the agent's
  // record or the Master, all counted on the stage's barrier
  auto fire = [&](int k, int p) {
    if (lane != 0) return;
    uint64_t* bar = &s_bar[k % kAttnDepth];
    const CUtensorMap* src_map = nullptr;
    int row = 0;
    bool pool_rows = false;
    if (p < hist) {
      const int64_t rk = pool_row_index(A.pool, a, layer, 0, p, A.err);
      if (rk >= 0) {
        src_map = &maps.pool;
        row = static_cast<int>(rk);
        pool_rows = true;
      }
    } else {
      const int t = p - hist;
      const int rec = __ldg(A.store.slot + (static_cast<int64_t>(a) * A.store.nl + sl) *
                                               A.rd.nb + t / A.rd.B);
      if (rec >= A.store.capacity) {
        atomicOr(A.err, err_bit(TD_ERR_INVALID_ARG));
      } else if (rec >= 0) {
        src_map = &maps.val_k;
        row = rec * A.rd.B + t % A.rd.B;
      } else {
        src_map = &maps.master_k;
        row = sl * S + t;
      }
    }
    mbar_arrive_expect_tx(bar, src_map ? 2u * TILE + A.tx_pad : A.tx_pad);
    if (!src_map) return;
    // the V rows: the pool's V half of the same page, or the V map of the same source
    const CUtensorMap* v_map = pool_rows ? &maps.pool
                             : (src_map == &maps.val_k ? &maps.val_v : &maps.master_v);
    const int v_row = pool_rows ? row + static_cast<int>(A.pool.num_pages) * P : row;
#pragma unroll
    for (int hh = 0; hh < HALVES; ++hh) {
      tma_box(s_k[k % kAttnDepth] + hh * BOX, src_map, h * D + hh * 64, row, bar);
      tma_box(s_v[k % kAttnDepth] + hh * BOX, v_map, h * D + hh * 64, v_row, bar);
    }
  };

  // this lane's query values: head gid of the group, dims kc*16 + tig*2 + {0, 1, 8, 9}
  // (the B operand of S^T = K Q^T: k = dims, n = query heads), read again per segment
  const bool qlive = gid < A.G;
  const uint16_t* qrow = A.q + ((static_cast<int64_t>(li) * A.n_list + A.x0 + x) * A.nq +
                                h * A.G + (qlive ? gid : 0)) * D;
  uint32_t qhi[KCH][2], qlo[KCH][2];
  bool two = false;
  // fragments of the segment's query: as given (history) or turned by R(-off_aj) (block j)
  auto build_q = [&](int seg) {
    float qraw[KCH][4], v[KCH][4];
#pragma unroll
    for (int kc = 0; kc < KCH; ++kc) {
      const uint32_t w0 = __ldg(reinterpret_cast<const unsigned int*>(qrow + kc * 16 + tig * 2));
      const uint32_t w1 = __ldg(reinterpret_cast<const unsigned int*>(qrow + kc * 16 + tig * 2 + 8));
      qraw[kc][0] = qlive ? bf_lo(w0) : 0.0f;
      qraw[kc][1] = qlive ? bf_hi(w0) : 0.0f;
      qraw[kc][2] = qlive ? bf_lo(w1) : 0.0f;
      qraw[kc][3] = qlive ? bf_hi(w1) : 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[kc][i] = qraw[kc][i];
    }
    two = seg >= 0;
    if (two) {
      const float* cs = A.rd.cos_t + static_cast<int64_t>(a * A.rd.M + seg) * (D / 2);
      const float* sn = A.rd.sin_t + static_cast<int64_t>(a * A.rd.M + seg) * (D / 2);
#pragma unroll
      for (int kc = 0; kc < KCH / 2; ++kc)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int f = kc * 16 + tig * 2 + (i & 1) + (i >> 1) * 8;
          const float cf = __ldg(cs + f), sf = __ldg(sn + f);
          const float x0 = qraw[kc][i], x1 = qraw[kc + KCH / 2][i];
          v[kc][i] = __fmaf_rn(x0, cf, __fmul_rn(x1, sf));
          v[kc + KCH / 2][i] = __fmaf_rn(x1, cf, -__fmul_rn(x0, sf));
        }
    }
#pragma unroll
    for (int kc = 0; kc < KCH; ++kc) {
      float hv[4], lv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hv[i] = __uint_as_float(static_cast<uint32_t>(bf16_bits(v[kc][i])) << 16);
        lv[i] = __fsub_rn(v[kc][i], hv[i]);
      }
      qhi[kc][0] = pack_bf2(hv[0], hv[1]);
      qhi[kc][1] = pack_bf2(hv[2], hv[3]);
      qlo[kc][0] = pack_bf2(lv[0], lv[1]);
      qlo[kc][1] = pack_bf2(lv[2], lv[3]);
    }
  };

  // O^T of the head group: oacc[mt] = dims mt*16 + gid (+8) x heads 2*tig, 2*tig + 1
  float oacc[KCH][4];
#pragma unroll
  for (int mt = 0; mt < KCH; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};   // heads 2*tig, 2*tig + 1
  float l_part[2] = {0.0f, 0.0f};            // this lane's share of their sums

  // prologue: the first stages in flight
  int ipos = p0, issued = 0;
  for (int k = 0; k < kAttnDepth && ipos < p1; ++k) {
    fire(k, ipos);
    ipos = stage_end(ipos);
    ++issued;
  }
  int cseg = -2;
  int cpos = p0;
  bool failed = false;
  // ldmatrix rows: K as the A operand (rows = positions), V transposed (rows = positions
  // of the transposed tile); which 8x8 matrix this lane addresses
  const int k_row = ((lane >> 3) & 1) * 8 + (lane & 7), k_c = lane >> 4;
  const int v_row = (lane >> 4) * 8 + (lane & 7), v_c = (lane >> 3) & 1;
  for (int k = 0; cpos < p1; ++k) {
    const int cend = stage_end(cpos);
    const int n = cend - cpos;
    const int buf = k % kAttnDepth;
    if (!mbar_wait_bounded(&s_bar[buf], (k / kAttnDepth) & 1)) {
      failed = true;
      if (lane == 0) atomicOr(A.err, err_bit(TD_ERR_DEVICE_TIMEOUT));
      for (int k2 = k; k2 < issued; ++k2)   // the copies this unit issued, stage k's too
        mbar_wait_bounded(&s_bar[k2 % kAttnDepth], (k2 / kAttnDepth) & 1);
      break;
    }
    if (n < kAttnStage) {
      // the boxes brought 16 rows; those past the stage get weight 0 below, and their V is
      // cleared so that no stray value can reach the sums
      for (int i = lane; i < (kAttnStage - n) * (TILE / kAttnStage / 16); i += 32) {
        const int r = n + i / (TILE / kAttnStage / 16);
        const int cc = i % (TILE / kAttnStage / 16);
        *reinterpret_cast<uint4*>(s_v[buf] + (cc >> 3) * BOX + swz(r, cc & 7)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    const int seg = segment(cpos);
    if (seg != cseg) {
      build_q(seg);
      cseg = seg;
    }
    // S^T = K Q^T: positions gid, gid + 8 x heads 2*tig, 2*tig + 1; four independent
    // chains (high / low part of the query x even / odd k-chunks)
    float sacc[4][4];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) sacc[ch][0] = sacc[ch][1] = sacc[ch][2] = sacc[ch][3] = 0.0f;
#pragma unroll
    for (int kc = 0; kc < KCH; ++kc) {
      uint32_t af[4];
      // chunk kc: box kc / 4, 16-byte chunks (kc % 4) * 2 + {0, 1} of the 128-byte row
      ldmatrix_x4(af, s_k[buf] + (kc >> 2) * BOX + swz(k_row, (kc & 3) * 2 + k_c));
      mma_bf16_full(sacc[kc & 1], af, qhi[kc][0], qhi[kc][1]);
      if (two) mma_bf16_full(sacc[2 + (kc & 1)], af, qlo[kc][0], qlo[kc][1]);
    }
    // scores (base 2) of (position r, head c): r = gid + 8 * (i >> 1), c = 2 * tig + (i & 1)
    float s2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool valid = 2 * tig + (i & 1) < A.G && gid + 8 * (i >> 1) < n;
      const float sc = __fadd_rn(__fadd_rn(sacc[0][i], sacc[1][i]),
                                 __fadd_rn(sacc[2][i], sacc[3][i]));
      s2[i] = valid ? sc * A.scale_log2 : -INFINITY;
    }
    float fac[2], p[4];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      float mx = fmaxf(s2[c2], s2[c2 + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float m_new = fmaxf(m_run[c2], mx);
      fac[c2] = m_run[c2] == -INFINITY ? 0.0f : exp2f(m_run[c2] - m_new);
      p[c2] = s2[c2] == -INFINITY ? 0.0f : exp2f(s2[c2] - m_new);
      p[c2 + 2] = s2[c2 + 2] == -INFINITY ? 0.0f : exp2f(s2[c2 + 2] - m_new);
      l_part[c2] = __fmaf_rn(l_part[c2], fac[c2], p[c2] + p[c2 + 2]);
      m_run[c2] = m_new;
    }
    // P^T as the B operand of O^T += V^T P^T (k = positions, n = heads): transposed
    // through shared memory (the stage's K tile, read completely by now), then split into
    // two bf16 parts like the query
    float (*s_pt)[kAttnGMax + 1] = reinterpret_cast<float (*)[kAttnGMax + 1]>(s_k[buf]);
    s_pt[gid][2 * tig] = p[0];
    s_pt[gid][2 * tig + 1] = p[1];
    s_pt[gid + 8][2 * tig] = p[2];
    s_pt[gid + 8][2 * tig + 1] = p[3];
    __syncwarp();
    const float pt[4] = {s_pt[2 * tig][gid], s_pt[2 * tig + 1][gid], s_pt[2 * tig + 8][gid],
                         s_pt[2 * tig + 9][gid]};
    float ph[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ph[i] = __uint_as_float(static_cast<uint32_t>(bf16_bits(pt[i])) << 16);
    const uint32_t bh0 = pack_bf2(ph[0], ph[1]), bh1 = pack_bf2(ph[2], ph[3]);
    const uint32_t bl0 = pack_bf2(__fsub_rn(pt[0], ph[0]), __fsub_rn(pt[1], ph[1]));
    const uint32_t bl1 = pack_bf2(__fsub_rn(pt[2], ph[2]), __fsub_rn(pt[3], ph[3]));
#pragma unroll
    for (int mt = 0; mt < KCH; ++mt) {
      uint32_t af[4];
      ldmatrix_x4_trans(af, s_v[buf] + (mt >> 2) * BOX + swz(v_row, (mt & 3) * 2 + v_c));
      oacc[mt][0] *= fac[0];
      oacc[mt][1] *= fac[1];
      oacc[mt][2] *= fac[0];
      oacc[mt][3] *= fac[1];
      mma_bf16_full(oacc[mt], af, bh0, bh1);
      mma_bf16_full(oacc[mt], af, bl0, bl1);
    }
    __syncwarp();   // this stage's buffers and s_pt are no longer read
    cpos = cend;
    if (ipos < p1) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fire(issued, ipos);
      __syncwarp();
      ipos = stage_end(ipos);
      ++issued;
    }
  }
  if (failed) return;
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    l_part[c2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[c2], 4);
    l_part[c2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[c2], 8);
    l_part[c2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[c2], 16);
  }
  // the partial of the group's G query heads only ([unit][G][D] and [unit][G][2])
  const int64_t unit = blockIdx.x;
  float* po = A.part_o + unit * A.G * D;
  const bool c0 = 2 * tig < A.G, c1 = 2 * tig + 1 < A.G;
#pragma unroll
  for (int mt = 0; mt < KCH; ++mt) {
    if (c0) {
      po[(2 * tig) * D + mt * 16 + gid] = oacc[mt][0];
      po[(2 * tig) * D + mt * 16 + gid + 8] = oacc[mt][2];
    }
    if (c1) {
      po[(2 * tig + 1) * D + mt * 16 + gid] = oacc[mt][1];
      po[(2 * tig + 1) * D + mt * 16 + gid + 8] = oacc[mt][3];
    }
  }
  if (gid == 0) {
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      if (2 * tig + c2 < A.G) {
        A.part_ml[(unit * A.G + 2 * tig + c2) * 2] = m_run[c2];
        A.part_ml[(unit * A.G + 2 * tig + c2) * 2 + 1] = l_part[c2];
      }
    }
  }
}

// One warp per (layer, agent, query head): merges the agent's units, normalises, writes
// the output row and the natural-log sum of exponentials of the scaled scores.
template <int D>
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs A, AttnList list) {
  pdl_wait();
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int64_t n_rows = static_cast<int64_t>(A.nl) * list.n * A.nq;
  if (w >= n_rows) return;
  const int gq = static_cast<int>(w % A.nq);
  const int x = static_cast<int>((w / A.nq) % list.n);
  const int li = static_cast<int>(w / (static_cast<int64_t>(A.nq) * list.n));
  const int h = gq / A.G, g = gq - h * A.G;
  // the agent's units: contiguous within (layer, kv head), long units before the split
  // layer, short ones from it on (after all the long units of the launch)
  const bool short_unit = li >= list.split;
  const int32_t* base = short_unit ? list.base2 : list.base;
  const int total = base[list.n];
  const int64_t first = short_unit ? static_cast<int64_t>(list.split) * A.g.H * list.base[list.n]
                                   : 0;
  const int lr = short_unit ? li - list.split : li;
  const int64_t u0 = first + (static_cast<int64_t>(lr) * A.g.H + h) * total + base[x];
  const int nu = base[x + 1] - base[x];
  auto unit_of = [&](int i) { return u0 + i; };
  // the units' maxima and sums a lane per unit (batches of 32), so that their loads are in
  // flight together; then the weighted outputs, eight units' loads at a time
  float mx = -INFINITY;
  for (int i0 = 0; i0 < nu; i0 += 32) {
    const int i = i0 + lane;
    if (i < nu) mx = fmaxf(mx, A.part_ml[(unit_of(i) * A.G + g) * 2]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  float l = 0.0f, acc[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.0f;
  for (int i0 = 0; i0 < nu; i0 += 32) {
    const int i = i0 + lane;
    float wgt = 0.0f;
    if (i < nu) {
      const int64_t unit = unit_of(i);
      const float m = A.part_ml[(unit * A.G + g) * 2];
      wgt = m == -INFINITY ? 0.0f : exp2f(m - mx);
      l = __fmaf_rn(A.part_ml[(unit * A.G + g) * 2 + 1], wgt, l);
    }
    const int nb = min(32, nu - i0);
#pragma unroll 8
    for (int j = 0; j < nb; ++j) {
      const float wj = __shfl_sync(0xFFFFFFFFu, wgt, j);
      const float* po = A.part_o + (unit_of(i0 + j) * A.G + g) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(po);
        acc[0] = __fmaf_rn(q4.x, wj, acc[0]);
        acc[1] = __fmaf_rn(q4.y, wj, acc[1]);
        acc[2] = __fmaf_rn(q4.z, wj, acc[2]);
        acc[3] = __fmaf_rn(q4.w, wj, acc[3]);
      } else {
        const float2 q2 = *reinterpret_cast<const float2*>(po);
        acc[0] = __fmaf_rn(q2.x, wj, acc[0]);
        acc[1] = __fmaf_rn(q2.y, wj, acc[1]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
  const int64_t row = (static_cast<int64_t>(li) * A.n_list + A.x0 + x) * A.nq + gq;
  const float inv = 1.0f / l;
#pragma unroll
  for (int d = 0; d < DPL; ++d) A.out[row * D + lane * DPL + d] = acc[d] * inv;
  if (lane == 0 && A.lse) A.lse[row] = (mx + log2f(l)) * 0.69314718055994530942f;
}

template <int D, bool kFromPool>
static cudaError_t run_attn(const AttnArgs& a, const AttnList& list, const AttnMaps& maps,
                            cudaStream_t st) {
  const int64_t units = static_cast<int64_t>(list.split) * a.g.H * list.base[list.n] +
                        static_cast<int64_t>(a.nl - list.split) * a.g.H * list.base2[list.n];
  if (units == 0) return cudaSuccess;
  cudaError_t e = launch_after(attn_unit_kernel<D, kFromPool>, static_cast<unsigned>(units), 32,
                               0, st, a, list, maps);
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.nl) * list.n * a.nq;
  return launch_after(attn_combine_kernel<D>, static_cast<unsigned>((rows + 3) / 4), 128, 0, st,
                      a, list);
}

cudaError_t launch_attention(const AttnArgs& a, const AttnList& list, const AttnMaps& maps,
                             bool from_pool, cudaStream_t st) {
  if (a.g.D == 128)
    return from_pool ? run_attn<128, true>(a, list, maps, st)
                     : run_attn<128, false>(a, list, maps, st);
  if (a.g.D == 64)
    return from_pool ? run_attn<64, true>(a, list, maps, st)
                     : run_attn<64, false>(a, list, maps, st);
  return cudaErrorInvalidValue;
}

}  // namespace td
