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
// Work unit = (layer, kv head, agent, 512 positions of the agent's context), one warp:
//   - each position's K and V rows of the head (D bf16 each) are staged in shared memory
//     by cp.async.bulk, 16 positions a stage, three stages in flight on an mbarrier ring.
//     Every wait is bounded: on time-out the unit records TD_ERR_DEVICE_TIMEOUT, waits
//     (bounded again) for the copies it issued and returns;
//   - QK^T on the tensor cores: mma.sync m16n8k16 bf16, the head group's G <= 8 query
//     heads as rows (rows G..15 zero). A rotated query is float32; it is split into a bf16
//     high part and a bf16 low part, two products per k-chunk, so each score keeps 16 bits
//     of the query (history queries are bf16 already: one product);
//   - online softmax in base 2 per query head; PV in float32 on the CUDA cores, each lane
//     owning D/32 dimensions of every query head's output;
//   - the unit writes its partial (max, sum, unnormalised output); attn_combine_kernel
//     merges an agent's units.
// The same kernel with every position read from the pages (kFromPool) is plain paged
// decode attention over a restored cache: the baseline the fusion replaces.
#include "td_device.cuh"

namespace td {

namespace {

constexpr unsigned kSpinLimit = 1u << 22;   // mbarrier polls before a unit gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
  for (unsigned it = 0; it < kSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Global -> shared copy by the bulk-copy (TMA) engine; completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D += A * B, m16n8k16, bf16 inputs, float32 accumulators. A rows g and g + 8 of the
// thread's fragment: a0 (row g, k 0-7 pair), a2 (row g, k 8-15 pair); rows g + 8 are zero.
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return static_cast<uint16_t>(pack_bf2(x, 0.0f) & 0xFFFFu);
}

}  // namespace

template <int D, bool kFromPool>
__global__ void __launch_bounds__(32)
attn_unit_kernel(AttnArgs A, AttnList list) {
  constexpr int DPL = D / 32;         // output dimensions per lane
  constexpr int KCH = D / 16;         // k-chunks of one q.k product
  constexpr int RS = D * 2 + 16;      // staged row stride in bytes (conflict-free ldmatrix)
  __shared__ __align__(128) unsigned char s_k[kAttnDepth][kAttnStage * RS];
  __shared__ __align__(128) unsigned char s_v[kAttnDepth][kAttnStage * RS];
  __shared__ __align__(16) float s_p[kAttnStage][kAttnGMax];
  __shared__ float s_f[kAttnGMax];
  __shared__ __align__(8) uint64_t s_bar[kAttnDepth];

  const int lane = threadIdx.x;
  const int gid = lane >> 2, tig = lane & 3;   // mma fragment row / column pair
  const int total = list.base[list.n];
  int64_t u = blockIdx.x;
  const int c = static_cast<int>(u % total);
  u /= total;
  const int h = static_cast<int>(u % A.g.H);
  const int li = static_cast<int>(u / A.g.H);
  int lo = 0, hi = list.n - 1;                 // the agent of unit c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (list.base[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  const int x = lo, a = list.a[x];
  const int S = A.rd.S, E = A.g.E;
  const int n_ctx = list.hist[x] + S;
  const int hist = kFromPool ? n_ctx : list.hist[x];   // positions read from the pages
  const int p0 = (c - list.base[x]) * kAttnChunk;
  const int p1 = min(p0 + kAttnChunk, n_ctx);
  const int layer = A.layer_begin + li, sl = A.sl0 + li;

  if (lane < kAttnDepth) mbar_init(&s_bar[lane], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();

  // the stage that starts at position p: at most 16 positions of one segment (the history,
  // or one shared block: the query's rotation is constant within a segment)
  auto stage_end = [&](int p) {
    int seg_end = hist;
    if (p >= hist) {
      const int j = __ldg(A.rd.tok_block + (p - hist));
      seg_end = hist + (j + 1 < A.rd.M ? __ldg(A.rd.blk_start + j + 1) : S);
    }
    return min(min(p + kAttnStage, seg_end), p1);
  };
  auto segment = [&](int p) { return p < hist ? -1 : __ldg(A.rd.tok_block + (p - hist)); };

  // lanes 0-15 fetch the K rows, lanes 16-31 the V rows of the stage's positions
  auto issue = [&](int k, int p) {
    const int n = stage_end(p) - p;
    const int tk = lane & 15, kv = lane >> 4;
    const uint16_t* src = nullptr;
    if (tk < n) {
      const int pos = p + tk;
      if (pos < hist) {
        const int64_t row = pool_row_index(A.pool, a, layer, kv, pos, A.err);
        if (row >= 0) src = A.pool.base + row * E + h * D;
      } else {
        const int t = pos - hist;
        const int rec = __ldg(A.store.slot +
                              (static_cast<int64_t>(a) * A.store.nl + sl) * A.rd.nb + t / A.rd.B);
        if (rec >= A.store.capacity) {
          atomicOr(A.err, err_bit(TD_ERR_INVALID_ARG));
        } else if (rec >= 0) {
          src = (kv ? A.store.val_v : A.store.val_k) +
                (static_cast<int64_t>(rec) * A.rd.B + t % A.rd.B) * E + h * D;
        } else {
          src = (kv ? A.store.master_v : A.store.master_k) +
                (static_cast<int64_t>(sl) * S + t) * E + h * D;
        }
      }
    }
    const unsigned ok = __ballot_sync(0xFFFFFFFFu, src != nullptr);
    uint64_t* bar = &s_bar[k % kAttnDepth];
    if (lane == 0) mbar_arrive_expect_tx(bar, __popc(ok) * (D * 2));
    __syncwarp();
    if (src)
      bulk_g2s((kv ? s_v : s_k)[k % kAttnDepth] + tk * RS, src, D * 2, bar);
  };

  // this lane's query values: head row gid of the group, dims kc*16 + tig*2 + {0, 1, 8, 9}
  float qraw[KCH][4];
  {
    const bool live = gid < A.G;
    const uint16_t* qrow = A.q + ((static_cast<int64_t>(li) * A.n_list + A.x0 + x) * A.nq +
                                  h * A.G + (live ? gid : 0)) * D;
#pragma unroll
    for (int kc = 0; kc < KCH; ++kc) {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(qrow + kc * 16 + tig * 2);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(qrow + kc * 16 + tig * 2 + 8);
      qraw[kc][0] = live ? bf_lo(w0) : 0.0f;
      qraw[kc][1] = live ? bf_hi(w0) : 0.0f;
      qraw[kc][2] = live ? bf_lo(w1) : 0.0f;
      qraw[kc][3] = live ? bf_hi(w1) : 0.0f;
    }
  }
  uint32_t ahi[KCH][2], alo[KCH][2];
  bool two = false;
  // fragments of the segment's query: as given (history) or turned by R(-off_aj) (block j)
  auto build_q = [&](int seg) {
    float v[KCH][4];
#pragma unroll
    for (int kc = 0; kc < KCH; ++kc)
#pragma unroll
      for (int i = 0; i < 4; ++i) v[kc][i] = qraw[kc][i];
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
        const uint16_t hb = bf16_bits(v[kc][i]);
        hv[i] = __uint_as_float(static_cast<uint32_t>(hb) << 16);
        lv[i] = __fsub_rn(v[kc][i], hv[i]);
      }
      ahi[kc][0] = pack_bf2(hv[0], hv[1]);
      ahi[kc][1] = pack_bf2(hv[2], hv[3]);
      alo[kc][0] = pack_bf2(lv[0], lv[1]);
      alo[kc][1] = pack_bf2(lv[2], lv[3]);
    }
  };

  float o[kAttnGMax][DPL];
#pragma unroll
  for (int g = 0; g < kAttnGMax; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[g][d] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;   // of query head gid (four lanes each)

  // prologue: the first stages in flight
  int ipos = p0, issued = 0;
  for (int k = 0; k < kAttnDepth && ipos < p1; ++k) {
    issue(k, ipos);
    ipos = stage_end(ipos);
    ++issued;
  }
  int cseg = -2;
  int cpos = p0;
  bool failed = false;
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
    const int seg = segment(cpos);
    if (seg != cseg) {
      build_q(seg);
      cseg = seg;
    }
    // scores of head gid for positions nt*8 + tig*2 + {0, 1}
    float s2[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const unsigned char* kb = s_k[buf] + (nt * 8 + (lane & 7)) * RS + (lane >> 4) * 32 +
                                ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int cp = 0; cp < KCH / 2; ++cp) {
        uint32_t b[4];
        ldmatrix_x4(b, kb + cp * 64);
        mma_bf16(acc, ahi[2 * cp][0], ahi[2 * cp][1], b[0], b[1]);
        mma_bf16(acc, ahi[2 * cp + 1][0], ahi[2 * cp + 1][1], b[2], b[3]);
        if (two) {
          mma_bf16(acc, alo[2 * cp][0], alo[2 * cp][1], b[0], b[1]);
          mma_bf16(acc, alo[2 * cp + 1][0], alo[2 * cp + 1][1], b[2], b[3]);
        }
      }
#pragma unroll
      for (int col = 0; col < 2; ++col) {
        const bool valid = gid < A.G && nt * 8 + tig * 2 + col < n;
        s2[nt][col] = valid ? acc[col] * A.scale_log2 : -INFINITY;
      }
    }
    float smax = fmaxf(fmaxf(s2[0][0], s2[0][1]), fmaxf(s2[1][0], s2[1][1]));
    smax = fmaxf(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, 1));
    smax = fmaxf(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, 2));
    const float m_new = fmaxf(m_run, smax);
    const float fac = m_run == -INFINITY ? 0.0f : exp2f(m_run - m_new);
    float psum = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int col = 0; col < 2; ++col) {
        const float p = s2[nt][col] == -INFINITY ? 0.0f : exp2f(s2[nt][col] - m_new);
        psum += p;
        s_p[nt * 8 + tig * 2 + col][gid] = p;
      }
    psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 1);
    psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 2);
    l_run = __fmaf_rn(l_run, fac, psum);
    m_run = m_new;
    if (tig == 0) s_f[gid] = fac;
    __syncwarp();
    // PV: every query head's output over this lane's dimensions
#pragma unroll
    for (int g = 0; g < kAttnGMax; ++g) {
      const float f = s_f[g];
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[g][d] *= f;
    }
    const unsigned char* vb = s_v[buf] + lane * DPL * 2;
    for (int t = 0; t < n; ++t) {
      const float4 pa = *reinterpret_cast<const float4*>(&s_p[t][0]);
      const float4 pb = *reinterpret_cast<const float4*>(&s_p[t][4]);
      const float pg[kAttnGMax] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
      float vv[DPL];
      if constexpr (DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(vb + t * RS);
        vv[0] = bf_lo(w.x);
        vv[1] = bf_hi(w.x);
        vv[2] = bf_lo(w.y);
        vv[3] = bf_hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(vb + t * RS);
        vv[0] = bf_lo(w);
        vv[1] = bf_hi(w);
      }
#pragma unroll
      for (int g = 0; g < kAttnGMax; ++g)
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[g][d] = __fmaf_rn(pg[g], vv[d], o[g][d]);
    }
    __syncwarp();   // this stage's buffers and s_p, s_f are no longer read
    cpos = cend;
    if (ipos < p1) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(issued, ipos);
      ipos = stage_end(ipos);
      ++issued;
    }
  }
  if (failed) return;
  const int64_t unit = blockIdx.x;
  float* po = A.part_o + unit * kAttnGMax * D + lane * DPL;
#pragma unroll
  for (int g = 0; g < kAttnGMax; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) po[g * D + d] = o[g][d];
  if (tig == 0) {
    A.part_ml[(unit * kAttnGMax + gid) * 2] = m_run;
    A.part_ml[(unit * kAttnGMax + gid) * 2 + 1] = l_run;
  }
}

// One warp per (layer, agent, query head): merges the agent's units, normalises, writes
// the output row and the natural-log sum of exponentials of the scaled scores.
template <int D>
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs A, AttnList list) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int64_t n_rows = static_cast<int64_t>(A.nl) * list.n * A.nq;
  if (w >= n_rows) return;
  const int gq = static_cast<int>(w % A.nq);
  const int x = static_cast<int>((w / A.nq) % list.n);
  const int li = static_cast<int>(w / (static_cast<int64_t>(A.nq) * list.n));
  const int h = gq / A.G, g = gq - h * A.G;
  const int total = list.base[list.n];
  const int64_t u0 = (static_cast<int64_t>(li) * A.g.H + h) * total;
  float mx = -INFINITY;
  for (int c = list.base[x]; c < list.base[x + 1]; ++c)
    mx = fmaxf(mx, A.part_ml[((u0 + c) * kAttnGMax + g) * 2]);
  float l = 0.0f, acc[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.0f;
  for (int c = list.base[x]; c < list.base[x + 1]; ++c) {
    const int64_t unit = u0 + c;
    const float m = A.part_ml[(unit * kAttnGMax + g) * 2];
    const float wgt = m == -INFINITY ? 0.0f : exp2f(m - mx);
    l = __fmaf_rn(A.part_ml[(unit * kAttnGMax + g) * 2 + 1], wgt, l);
    const float* po = A.part_o + (unit * kAttnGMax + g) * D + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = __fmaf_rn(po[d], wgt, acc[d]);
  }
  const int64_t row = (static_cast<int64_t>(li) * A.n_list + A.x0 + x) * A.nq + gq;
  const float inv = 1.0f / l;
#pragma unroll
  for (int d = 0; d < DPL; ++d) A.out[row * D + lane * DPL + d] = acc[d] * inv;
  if (lane == 0 && A.lse) A.lse[row] = (mx + log2f(l)) * 0.69314718055994530942f;
}

template <int D, bool kFromPool>
static cudaError_t run_attn(const AttnArgs& a, const AttnList& list, cudaStream_t st) {
  const int64_t units = static_cast<int64_t>(a.nl) * a.g.H * list.base[list.n];
  if (units == 0) return cudaSuccess;
  attn_unit_kernel<D, kFromPool><<<static_cast<unsigned>(units), 32, 0, st>>>(a, list);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.nl) * list.n * a.nq;
  attn_combine_kernel<D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, st>>>(a, list);
  return cudaGetLastError();
}

cudaError_t launch_attention(const AttnArgs& a, const AttnList& list, bool from_pool,
                             cudaStream_t st) {
  if (a.g.D == 128)
    return from_pool ? run_attn<128, true>(a, list, st) : run_attn<128, false>(a, list, st);
  if (a.g.D == 64)
    return from_pool ? run_attn<64, true>(a, list, st) : run_attn<64, false>(a, list, st);
  return cudaErrorInvalidValue;
}

}  // namespace td
