// k_master.cu - stage 3a: Master choice (TokenDance review [R], Summary Method (3): keep the
// agent with the smallest deviation as the dense Master; §3c A2: the deviation score is
// chosen so that the Mirrors' diffs come out sparsest).
//
// One CTA per agent turns the agent's selection into a bitmask over the diff blocks (16
// or 32 tokens); the CTA that finishes last (a self-resetting counter; no CTA waits) gathers the
// masks and counts cost(m) = sum over i != m of popcount(mask_i | mask_m), one warp per
// candidate m; the smallest cost wins, ties to the lower index. Integer arithmetic only,
// so the result does not depend on the order of the additions.
#include "td_device.cuh"

namespace td {

__global__ void __launch_bounds__(1024)
pick_master_kernel(const int32_t* __restrict__ sel, int N, int S, int B, int k, int nbw,
                   int64_t* __restrict__ cost_out, int32_t* __restrict__ master,
                   uint32_t* gmask, int* done, uint32_t* err) {
  pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  unsigned* mask = reinterpret_cast<unsigned*>(smem_raw);            // [N][nbw] (last CTA)
  __shared__ int s_last;
  const int i = blockIdx.x;
  const int lane = threadIdx.x & 31;
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) mask[w] = 0u;
  __syncthreads();
  // the row ascends, so lanes that hit the same block are neighbours: only the first of a
  // run sets the bit (uniform trip count keeps the warp converged)
  const int32_t* row = sel + static_cast<int64_t>(i) * k;
  const int trips = (k + blockDim.x - 1) / blockDim.x;
  for (int it = 0; it < trips; ++it) {
    const int x = it * blockDim.x + threadIdx.x;
    int b = -1;
    if (x < k) {
      const int t = __ldg(row + x);
      if (t < 0 || t >= S) atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
      else b = t / B;
    }
    const int prev = __shfl_up_sync(0xFFFFFFFFu, b, 1);
    if (b >= 0 && (lane == 0 || prev != b)) atomicOr(&mask[b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nbw; w += blockDim.x) gmask[i * nbw + w] = mask[w];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(done, 1) == N - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) *done = 0;           // ready for the next call
  for (int x = threadIdx.x; x < N * nbw; x += blockDim.x) mask[x] = __ldcg(gmask + x);
  long long* cost = reinterpret_cast<long long*>(
      smem_raw + ((static_cast<size_t>(N) * nbw * 4 + 7) & ~size_t(7)));
  __syncthreads();
  const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int m = wid; m < N; m += nw) {
    long long c = 0;
    for (int x = lane; x < N * nbw; x += 32) {
      const int a = x / nbw, w = x - a * nbw;
      if (a != m) c += __popc(mask[a * nbw + w] | mask[m * nbw + w]);
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

cudaError_t launch_pick_master(const int32_t* sel, int N, int S, int B, int k, int64_t* cost,
                               int32_t* master, uint32_t* gmask, int* done, uint32_t* err,
                               cudaStream_t st) {
  const int nb = (S + B - 1) / B;
  const int nbw = (nb + 31) / 32;
  const size_t smem = ((static_cast<size_t>(N) * nbw * 4 + 7) & ~size_t(7)) + 8 * static_cast<size_t>(N);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(pick_master_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int threads = k >= 512 ? 1024 : 256;
  return launch_after(pick_master_kernel, static_cast<unsigned>(N), threads, smem, st, sel, N, S,
                      B, k, nbw, cost, master, gmask, done, err);
}

}  // namespace td
