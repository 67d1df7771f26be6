// k_master.cu - stage 3a: Master choice (TokenDance review [R], Summary Method (3): keep the
// agent with the smallest deviation as the dense Master; §3c A2: the deviation score is
// chosen so that the Mirrors' diffs come out sparsest).
//
// One CTA. Each agent's selection becomes a bitmask over the 16-token diff blocks (shared
// memory); cost(m) = sum over i != m of popcount(mask_i | mask_m), counted by one warp per
// candidate m; the smallest cost wins, ties to the lower index. Integer arithmetic only,
// so the result does not depend on the order of the additions.
#include "td_device.cuh"

namespace td {

__global__ void __launch_bounds__(1024)
pick_master_kernel(const int32_t* __restrict__ sel, int N, int S, int k, int nbw,
                   int64_t* __restrict__ cost_out, int32_t* __restrict__ master,
                   uint32_t* err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned* mask = reinterpret_cast<unsigned*>(smem_raw);                       // [N][nbw]
  long long* cost = reinterpret_cast<long long*>(smem_raw + ((static_cast<size_t>(N) * nbw * 4 + 7) & ~size_t(7)));
  for (int x = threadIdx.x; x < N * nbw; x += blockDim.x) mask[x] = 0u;
  __syncthreads();
  for (int64_t x = threadIdx.x; x < static_cast<int64_t>(N) * k; x += blockDim.x) {
    const int i = static_cast<int>(x / k);
    const int t = __ldg(sel + x);
    if (t < 0 || t >= S) {
      atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
      continue;
    }
    const int b = t / kDiffBlock;
    atomicOr(&mask[i * nbw + (b >> 5)], 1u << (b & 31));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int m = wid; m < N; m += nw) {
    long long c = 0;
    for (int x = lane; x < N * nbw; x += 32) {
      const int i = x / nbw, w = x - (x / nbw) * nbw;
      if (i != m) c += __popc(mask[i * nbw + w] | mask[m * nbw + w]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) {
      cost[m] = c;
      if (cost_out) cost_out[m] = c;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = 0;
    for (int m = 1; m < N; ++m)
      if (cost[m] < cost[best]) best = m;
    *master = best;
  }
}

cudaError_t launch_pick_master(const int32_t* sel, int N, int S, int k, int64_t* cost,
                               int32_t* master, uint32_t* err, cudaStream_t st) {
  const int nb = (S + kDiffBlock - 1) / kDiffBlock;
  const int nbw = (nb + 31) / 32;
  const size_t smem = ((static_cast<size_t>(N) * nbw * 4 + 7) & ~size_t(7)) + 8 * static_cast<size_t>(N);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(pick_master_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  pick_master_kernel<<<1, 1024, smem, st>>>(sel, N, S, k, nbw, cost, master, err);
  return cudaGetLastError();
}

}  // namespace td
