// k_select.cu - stage 2: key deviation at the check layer and per-agent top-k
// (TokenDance review [R], Summary Method (2): one key-difference analysis for the whole
// group at the check layer; its important positions are reused by all later layers).
//
// deviation_kernel: one warp per (agent, token). Lane l reads the 16-byte vectors
//   v = l, l+32, ... of the fresh row and of the reused row in the agent's page, adds
//   (a-b)^2 with fma in ascending element order, then the warp adds its 32 partial sums
//   with an xor butterfly (16, 8, 4, 2, 1). That order is part of the definition: the
//   selection is compared bit for bit.
// select_kernel: one CTA per agent, radix select on the float bits of the deviations
//   (non-negative, so the bits order like the values): four 8-bit digit passes find the
//   k-th largest value T; the output takes every token above T and the lowest-index
//   tokens equal to T, written in ascending token order by block-wide prefix sums.
#include "td_device.cuh"

namespace td {

__global__ void __launch_bounds__(256)
deviation_kernel(Geom g, RoundDev rd, PoolDev pool, int check_layer,
                 const uint16_t* __restrict__ kf, float* __restrict__ dev, uint32_t* err) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<int64_t>(rd.N) * rd.S) return;
  const int i = static_cast<int>(w / rd.S);
  const int t = static_cast<int>(w - static_cast<int64_t>(i) * rd.S);
  const int j = __ldg(rd.tok_block + t);
  const int pos = __ldg(rd.off + i * rd.M + j) + t - __ldg(rd.blk_start + j);
  // every lane computes the same address; only lane 0 may report a fault
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

// Block-wide exclusive scan of one 0/1 flag per thread (1024 threads); returns the
// prefix and writes the total to *total (shared).
__device__ __forceinline__ int block_scan_flag(bool f, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, f);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[wid] = __popc(bal);
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    int x = lane < nw ? warp_tot[lane] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nw) warp_tot[lane] = incl - x;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const int r = warp_tot[wid] + in_warp;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024)
select_kernel(const float* __restrict__ dev, int S, int k, int32_t* __restrict__ sel) {
  __shared__ unsigned hist[256];
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ unsigned s_prefix, s_mask;
  __shared__ int s_remaining;
  const int i = blockIdx.x;
  const unsigned* keys = reinterpret_cast<const unsigned*>(dev) + static_cast<int64_t>(i) * S;
  int32_t* out = sel + static_cast<int64_t>(i) * k;
  if (k <= 0) return;
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_mask = 0u;
    s_remaining = k;
  }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
    __syncthreads();
    const unsigned prefix = s_prefix, mask = s_mask;
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
      const unsigned key = __ldg(keys + t);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // warp 0..7: thread d' holds bin 255 - d'; inclusive scan from the top bin down
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
      const unsigned rem = static_cast<unsigned>(s_remaining);
      // all 8 warps must have written their totals before the cross-warp part
      asm volatile("bar.sync 1, 256;" ::: "memory");
      unsigned before = 0;
      for (int w = 0; w < wid; ++w) before += static_cast<unsigned>(warp_tot[w]);
      incl += before;
      const unsigned excl = incl - x;
      if (excl < rem && incl >= rem) {
        s_prefix = prefix | (static_cast<unsigned>(d) << shift);
        s_mask = mask | (255u << shift);
        s_remaining = static_cast<int>(rem - excl);
      }
    }
    __syncthreads();
  }
  const unsigned T = s_prefix;
  const int need_eq = s_remaining;  // tokens equal to T to take, lowest index first
  int base_out = 0, eq_seen = 0;
  for (int c0 = 0; c0 < S; c0 += blockDim.x) {
    const int t = c0 + threadIdx.x;
    const unsigned key = t < S ? __ldg(keys + t) : 0u;
    const bool gt = t < S && key > T;
    const bool eq = t < S && key == T;
    const int eq_rank = block_scan_flag(eq, warp_tot, &s_total);
    const int eq_tot = s_total;
    const bool take = gt || (eq && eq_seen + eq_rank < need_eq);
    const int pos = block_scan_flag(take, warp_tot, &s_total);
    if (take) out[base_out + pos] = t;
    base_out += s_total;
    eq_seen += eq_tot;
    __syncthreads();
  }
}

cudaError_t launch_deviation(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                             int check_layer, const uint16_t* k_fresh, float* dev,
                             uint32_t* err, cudaStream_t st) {
  const int64_t warps = static_cast<int64_t>(rd.N) * rd.S;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  deviation_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(g, rd, pool, check_layer,
                                                                  k_fresh, dev, err);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* dev, int N, int S, int k, int32_t* sel,
                          cudaStream_t st) {
  if (k <= 0 || N <= 0) return cudaSuccess;
  select_kernel<<<N, 1024, 0, st>>>(dev, S, k, sel);
  return cudaGetLastError();
}

}  // namespace td
