// k_variants.cu - the variant readings of two steps (TokenDance review [R], Summary Method
// (2) and (3) leave both open):
//   master by least total deviation: the agent whose selected tokens deviate least in
//     total; one warp per agent sums its k deviations in float64 in a fixed order (addend
//     r to lane r mod 32, lanes ascending, then an xor tree 16..1), one thread takes the
//     argmin (ties to the lower agent);
//   one group-wide important set: the group deviation of token t is the float32 sum of
//     the agents' deviations in agent order; its top-k (the same radix select as the
//     per-agent set) becomes every agent's selection.
#include "td_device.cuh"

namespace td {

__global__ void __launch_bounds__(1024)
min_dev_master_kernel(const int32_t* __restrict__ sel, const float* __restrict__ dev, int N,
                      int S, int k, double* __restrict__ score, int32_t* __restrict__ master,
                      uint32_t* err) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int i = wid; i < N; i += nw) {
    double acc = 0.0;
    for (int r = lane; r < k; r += 32) {
      const int t = __ldg(sel + static_cast<int64_t>(i) * k + r);
      if (t < 0 || t >= S) {
        atomicOr(err, err_bit(TD_ERR_INVALID_ARG));
        continue;
      }
      acc = __dadd_rn(acc, static_cast<double>(__ldg(dev + static_cast<int64_t>(i) * S + t)));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = __dadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if (lane == 0) score[i] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = -1;
    for (int i = 0; i < N; ++i) {
      const double v = score[i];
      if (isnan(v) || isinf(v)) {
        atomicOr(err, err_bit(TD_ERR_NONFINITE));
        continue;
      }
      if (best < 0 || v < score[best]) best = i;
    }
    *master = best < 0 ? 0 : best;
  }
}

__global__ void __launch_bounds__(256)
group_dev_kernel(const float* __restrict__ dev, int N, int S, float* __restrict__ g) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= S) return;
  float s = 0.0f;
  for (int i = 0; i < N; ++i) s = __fadd_rn(s, __ldg(dev + static_cast<int64_t>(i) * S + t));
  g[t] = s;
}

__global__ void __launch_bounds__(256)
broadcast_rows_kernel(int32_t* __restrict__ sel, int N, int k) {
  const int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x >= static_cast<int64_t>(N - 1) * k) return;
  const int r = static_cast<int>(x % k);
  sel[k + x] = sel[r];
}

cudaError_t launch_min_dev_master(const int32_t* sel, const float* dev, int N, int S, int k,
                                  double* score, int32_t* master, uint32_t* err,
                                  cudaStream_t st) {
  min_dev_master_kernel<<<1, 1024, 0, st>>>(sel, dev, N, S, k, score, master, err);
  return cudaGetLastError();
}

cudaError_t launch_check_select_group(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                      int check_layer, const uint16_t* k_fresh, float* dev,
                                      float* gdev, int k, int32_t* sel, uint32_t* err,
                                      cudaStream_t st) {
  cudaError_t e = launch_deviation(g, rd, pool, check_layer, k_fresh, dev, err, st);
  if (e != cudaSuccess) return e;
  group_dev_kernel<<<(rd.S + 255) / 256, 256, 0, st>>>(dev, rd.N, rd.S, gdev);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (k <= 0) return cudaSuccess;
  if ((e = launch_select(gdev, 1, rd.S, k, sel, st)) != cudaSuccess) return e;
  const int64_t rest = static_cast<int64_t>(rd.N - 1) * k;
  if (rest > 0) {
    broadcast_rows_kernel<<<static_cast<unsigned>((rest + 255) / 256), 256, 0, st>>>(sel, rd.N, k);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace td
