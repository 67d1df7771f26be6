// k_select.cu - stage 2: key deviation at the check layer and per-agent top-k
// (TokenDance review [R], Summary Method (2): one key-difference analysis for the whole
// group at the check layer; its important positions are reused by all later layers).
//
// deviation_kernel: one warp per (agent, token) computes the squared deviation - lane l
//   reads the 16-byte vectors v = l, l+32, ... of the fresh row and of the reused row in
//   the agent's page, adds (a-b)^2 with fma in ascending element order, then the warp adds
//   its 32 partial sums with an xor butterfly (16, 8, 4, 2, 1). That order is part of the
//   definition: the selection is compared bit for bit.
// select_kernel: one CTA per agent, radix select on the float bits of the deviations
//   (non-negative, so the bits order like the values): four 8-bit digit passes find the
//   k-th largest value T; the output takes every token above T and the lowest-index
//   tokens equal to T, in ascending token order (one block scan over contiguous ranges).
#include "td_device.cuh"

namespace td {

// Squared deviation of one (agent, token) by one warp, in the fixed order: lane l takes
// the 16-byte vectors l, l+32, ... and adds (a-b)^2 with fma, then xor tree 16..1.
__device__ __forceinline__ void deviation_token(const Geom& g, const RoundDev& rd,
                                                const PoolDev& pool, int check_layer,
                                                const uint16_t* __restrict__ kf,
                                                float* __restrict__ dev, int64_t w, int lane,
                                                uint32_t* err) {
  const int i = static_cast<int>(w / rd.S);
  const int t = static_cast<int>(w - static_cast<int64_t>(i) * rd.S);
  const int j = __ldg(rd.tok_block + t);
  const int pos = __ldg(rd.off + i * rd.M + j) + t - __ldg(rd.blk_start + j);
  // every lane computes the same address; only lane 0 reports a fault
  const int lp = pool.p_shift >= 0 ? (pos >> pool.p_shift) : pos / pool.P;
  int32_t page = -1;
  if (lp < pool.max_lp) page = __ldg(pool.bt + static_cast<int64_t>(i) * pool.max_lp + lp);
  if (page < 0 || page >= pool.num_pages) {
    if (lane == 0) {
      atomicOr(err, err_bit(TD_ERR_UNMAPPED_PAGE));
      dev[w] = 0.0f;
    }
    return;
  }
  const uint16_t* reused =
      pool.base + (((static_cast<int64_t>(check_layer) * 2) * pool.num_pages + page) * pool.P +
                   (pos - lp * pool.P)) * g.E;
  const uint16_t* fresh = kf + w * g.E;
  float acc = 0.0f;
  for (int v = lane; v < (g.E >> 3); v += 32) {
    float a[8], b[8];
    unpack8(ldg16(fresh + v * 8), a);
    unpack8(ld16(reused + v * 8), b);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float d = __fsub_rn(a[q], b[q]);
      acc = __fmaf_rn(d, d, acc);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
  if (lane == 0) {
    dev[w] = acc;
    if (!isfinite(acc)) atomicOr(err, err_bit(TD_ERR_NONFINITE));
  }
}

__global__ void __launch_bounds__(256)
deviation_kernel(Geom g, RoundDev rd, PoolDev pool, int check_layer,
                 const uint16_t* __restrict__ kf, float* __restrict__ dev, uint32_t* err) {
  pdl_wait();
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= static_cast<int64_t>(rd.N) * rd.S) return;
  deviation_token(g, rd, pool, check_layer, kf, dev, w, threadIdx.x & 31, err);
}

// Radix top-k of one agent's deviations by the whole CTA (any multiple of 32 threads, at
// least 256). Keys are read through L2 (they may have been written by other CTAs of the
// same launch).
__device__ void select_agent(const float* dev_i, int S, int k, int32_t* out, unsigned* hist,
                             int* warp_tot, int* s_total, unsigned* s_prefix, unsigned* s_mask,
                             int* s_remaining) {
  const unsigned* keys = reinterpret_cast<const unsigned*>(dev_i);
  if (k <= 0) return;
  if (threadIdx.x == 0) {
    *s_prefix = 0u;
    *s_mask = 0u;
    *s_remaining = k;
  }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
    __syncthreads();
    const unsigned prefix = *s_prefix, mask = *s_mask;
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
      const unsigned key = __ldcg(keys + t);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // threads 0..255: thread d' holds bin 255 - d'; inclusive scan from the top bin down
    if (threadIdx.x < 256) {
      const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
      const int d = 255 - threadIdx.x;
      const unsigned x = hist[d];
      unsigned incl = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) warp_tot[wid] = static_cast<int>(incl);
      // read before the barrier: the one thread that finds the digit rewrites it after
      const unsigned rem = static_cast<unsigned>(*s_remaining);
      // all 8 warps must have written their totals before the cross-warp part
      asm volatile("bar.sync 1, 256;" ::: "memory");
      unsigned before = 0;
      for (int w = 0; w < wid; ++w) before += static_cast<unsigned>(warp_tot[w]);
      incl += before;
      const unsigned excl = incl - x;
      if (excl < rem && incl >= rem) {
        *s_prefix = prefix | (static_cast<unsigned>(d) << shift);
        *s_mask = mask | (255u << shift);
        *s_remaining = static_cast<int>(rem - excl);
      }
    }
    __syncthreads();
  }
  const unsigned T = *s_prefix;
  const int need_eq = *s_remaining;  // tokens equal to T to take, lowest index first
  // each thread owns a contiguous range of tokens; one block scan of its (above T, equal
  // to T) counts gives where its selected tokens go, in ascending token order
  const int per = (S + blockDim.x - 1) / blockDim.x;
  const int r0 = min(S, static_cast<int>(threadIdx.x) * per), r1 = min(S, r0 + per);
  unsigned long long cnt = 0;
  for (int t = r0; t < r1; ++t) {
    const unsigned key = __ldcg(keys + t);
    cnt += key > T ? (1ull << 32) : (key == T ? 1ull : 0ull);
  }
  unsigned long long* wsum = reinterpret_cast<unsigned long long*>(hist);  // reuse
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();                   // the histogram is no longer read
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  unsigned long long before = 0;
  for (int w = 0; w < wid && w < nw; ++w) before += wsum[w];
  const unsigned long long excl = before + incl - cnt;
  const int pre_gt = static_cast<int>(excl >> 32);
  int eq_seen = static_cast<int>(excl & 0xFFFFFFFFull);
  int pos = pre_gt + min(eq_seen, need_eq);
  for (int t = r0; t < r1; ++t) {
    const unsigned key = __ldcg(keys + t);
    if (key > T) {
      out[pos++] = t;
    } else if (key == T) {
      if (eq_seen < need_eq) out[pos++] = t;
      ++eq_seen;
    }
  }
  __syncthreads();                   // shared scratch may be reused by the caller
}

__global__ void __launch_bounds__(1024)
select_kernel(const float* __restrict__ dev, int S, int k, int32_t* __restrict__ sel) {
  pdl_wait();
  __shared__ __align__(16) unsigned hist[256];
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_remaining;
  __shared__ unsigned s_prefix, s_mask;
  const int i = blockIdx.x;
  select_agent(dev + static_cast<int64_t>(i) * S, S, k, sel + static_cast<int64_t>(i) * k,
               hist, warp_tot, &s_total, &s_prefix, &s_mask, &s_remaining);
}

cudaError_t launch_deviation(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                             int check_layer, const uint16_t* k_fresh, float* dev,
                             uint32_t* err, cudaStream_t st) {
  const int64_t warps = static_cast<int64_t>(rd.N) * rd.S;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  return launch_after(deviation_kernel, static_cast<unsigned>(blocks), 256, 0, st, g, rd, pool,
                      check_layer, k_fresh, dev, err);
}

cudaError_t launch_select(const float* dev, int N, int S, int k, int32_t* sel,
                          cudaStream_t st) {
  if (k <= 0 || N <= 0) return cudaSuccess;
  return launch_after(select_kernel, static_cast<unsigned>(N), 1024, 0, st, dev, S, k, sel);
}

cudaError_t launch_check_select(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                int check_layer, const uint16_t* k_fresh, float* dev, int k,
                                int32_t* sel, uint32_t* err, cudaStream_t st) {
  cudaError_t e = launch_deviation(g, rd, pool, check_layer, k_fresh, dev, err, st);
  if (e != cudaSuccess) return e;
  return launch_select(dev, rd.N, rd.S, k, sel, st);
}

}  // namespace td
