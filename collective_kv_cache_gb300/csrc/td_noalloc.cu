// td_noalloc.cu - td_check_select_noalloc: the check-layer selection for callers that cannot
// allocate device memory (for example code running under an allocator that forbids
// cudaMalloc, or a caller that must not grow its memory footprint after start-up).
//
// It runs the same deviation and top-k kernels as td_check_select, but its scratch - the
// round's copied descriptor, offsets and token tables, the deviations and the error word -
// lives in one file-scope device array of fixed size instead of a context's allocations.
// Every GPU that loads the library holds that array until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "td.h"
#include "td_internal.h"

namespace td {
namespace {

// Fixed maxima of the scratch (the entry point rejects anything larger).
constexpr int kNaMaxAgents = 256;
constexpr int kNaMaxBlocks = 256;
constexpr int kNaMaxAgentBlocks = 16384;       // N * M
constexpr int kNaMaxShared = 65536;            // S
constexpr int64_t kNaMaxDev = int64_t(1) << 20;  // N * S deviations (4 MiB)

// Byte layout of the scratch; each region starts on a 256-byte boundary.
constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kOffErr = 0;
constexpr size_t kOffLen = align256(kOffErr + 4);
constexpr size_t kOffHist = align256(kOffLen + 4 * kNaMaxBlocks);
constexpr size_t kOffPerm = align256(kOffHist + 4 * kNaMaxAgents);
constexpr size_t kOffOff = align256(kOffPerm + 4 * size_t(kNaMaxAgentBlocks));
constexpr size_t kOffStart = align256(kOffOff + 4 * size_t(kNaMaxAgentBlocks));
constexpr size_t kOffTok = align256(kOffStart + 4 * kNaMaxBlocks);
constexpr size_t kOffDev = align256(kOffTok + 4 * size_t(kNaMaxShared));
constexpr size_t kScratchBytes = align256(kOffDev + 4 * size_t(kNaMaxDev));

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

// Host code cannot use g_select_scratch as an address: it is a host-side stand-in. The
// device address is looked up with the device current and kept, per device, together with
// the CUDA context it belongs to: after a device reset the device has a new context (and
// the array a new address), so the address is looked up again.
constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
unsigned char* g_addr[kMaxDevices] = {};
void* g_addr_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

void* current_context() {
  CUcontext c = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

cudaError_t scratch_address(unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  void* ctx = current_context();
  if (!g_addr[dev] || !ctx || g_addr_ctx[dev] != ctx) {
    // the lookup also creates the device's context if none is current yet
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<unsigned char*>(p);
    g_addr_ctx[dev] = current_context();
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

// Offsets, block starts and the token -> block table from the copied round descriptor.
__global__ void __launch_bounds__(256) noalloc_tables_kernel(int N, int M) {
  unsigned char* base = g_select_scratch;
  const int32_t* len = reinterpret_cast<const int32_t*>(base + kOffLen);
  const int32_t* hist = reinterpret_cast<const int32_t*>(base + kOffHist);
  const int32_t* perm = reinterpret_cast<const int32_t*>(base + kOffPerm);
  int32_t* off = reinterpret_cast<int32_t*>(base + kOffOff);
  int32_t* start = reinterpret_cast<int32_t*>(base + kOffStart);
  int32_t* tok = reinterpret_cast<int32_t*>(base + kOffTok);
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    int pos = hist[i];
    for (int q = 0; q < M; ++q) {
      const int j = perm[i * M + q];
      off[i * M + j] = pos;
      pos += len[j];
    }
  }
  if (threadIdx.x == 0) {
    int s = 0;
    for (int j = 0; j < M; ++j) {
      start[j] = s;
      s += len[j];
    }
  }
  __syncthreads();
  for (int j = 0; j < M; ++j)
    for (int u = threadIdx.x; u < len[j]; u += blockDim.x) tok[start[j] + u] = j;
}

}  // namespace
}  // namespace td

using namespace td;

extern "C" td_status td_check_select_noalloc(const td_shape* shape, const td_round* r,
                                             int32_t check_layer, const td_paged* pool,
                                             const void* k_fresh, int32_t recompute_pct,
                                             int32_t* sel, int32_t* k_out,
                                             uint32_t* err_bits_out, void* stream) {
  if (!shape || !r || !pool || !k_fresh || !k_out || !r->block_len || !r->hist_len ||
      !r->perm || !pool->base || !pool->block_table)
    return TD_ERR_INVALID_ARG;
  const td_shape& s = *shape;
  if (s.n_layers < 1 || s.n_kv_heads < 1 || s.head_dim < 16 || s.head_dim % 16 != 0 ||
      s.page_size < 1 || (s.diff_block != kDiffBlock && s.diff_block != kMaxDiffBlock))
    return TD_ERR_INVALID_ARG;   // the selection does not depend on the diff block
  const int64_t E = static_cast<int64_t>(s.n_kv_heads) * s.head_dim;
  if (E > 2048) return TD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_fresh) & 15u) || (reinterpret_cast<uintptr_t>(pool->base) & 15u))
    return TD_ERR_INVALID_ARG;
  if (check_layer < 0 || check_layer >= s.n_layers || recompute_pct < 0 || recompute_pct > 100 ||
      pool->num_pages < 1 || pool->max_pages_per_agent < 1)
    return TD_ERR_INVALID_ARG;
  const int N = r->n_agents, M = r->n_blocks;
  if (N < 1 || M < 1) return TD_ERR_INVALID_ARG;
  if (N > kNaMaxAgents || M > kNaMaxBlocks || static_cast<int64_t>(N) * M > kNaMaxAgentBlocks)
    return TD_ERR_SCRATCH_LIMIT;
  int64_t S = 0;
  for (int j = 0; j < M; ++j) {
    if (r->block_len[j] < 1) return TD_ERR_INVALID_ARG;
    S += r->block_len[j];
  }
  if (S > kNaMaxShared || static_cast<int64_t>(N) * S > kNaMaxDev) return TD_ERR_SCRATCH_LIMIT;
  for (int i = 0; i < N; ++i) {
    if (r->hist_len[i] < 0) return TD_ERR_INVALID_ARG;
    if ((static_cast<int64_t>(r->hist_len[i]) + S - 1) / s.page_size >= pool->max_pages_per_agent)
      return TD_ERR_INVALID_ARG;
    unsigned char seen[kNaMaxBlocks] = {};
    for (int q = 0; q < M; ++q) {
      const int j = r->perm[static_cast<int64_t>(i) * M + q];
      if (j < 0 || j >= M || seen[j]) return TD_ERR_INVALID_ARG;
      seen[j] = 1;
    }
  }
  const int k = static_cast<int>((static_cast<int64_t>(recompute_pct) * S + 99) / 100);
  if (k > 0 && !sel) return TD_ERR_INVALID_ARG;

  unsigned char* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return TD_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(base + kOffErr);
  // The round descriptor is copied from the caller's host arrays on the stream: from
  // pageable memory the copy has read them when it returns, from page-locked memory it
  // may read them later (the caller keeps them unchanged until the stream passes here).
  if (cudaMemsetAsync(err, 0, 4, st) != cudaSuccess ||
      cudaMemcpyAsync(base + kOffLen, r->block_len, 4 * size_t(M), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(base + kOffHist, r->hist_len, 4 * size_t(N), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(base + kOffPerm, r->perm, 4 * size_t(N) * M, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return TD_ERR_CUDA;
  noalloc_tables_kernel<<<1, 256, 0, st>>>(N, M);
  if (cudaGetLastError() != cudaSuccess) return TD_ERR_CUDA;

  Geom g;
  g.H = s.n_kv_heads;
  g.D = s.head_dim;
  g.E = static_cast<int>(E);
  g.half = s.head_dim / 2;
  g.vpt = static_cast<int>(E / 16);
  RoundDev rd;
  rd.N = N;
  rd.M = M;
  rd.S = static_cast<int>(S);
  rd.B = s.diff_block;
  rd.nb = static_cast<int>((S + s.diff_block - 1) / s.diff_block);
  rd.nt = static_cast<int>((S + kTile - 1) / kTile);
  rd.off = reinterpret_cast<const int32_t*>(base + kOffOff);
  rd.cos_t = nullptr;  // the deviation pass turns nothing
  rd.sin_t = nullptr;
  rd.tok_block = reinterpret_cast<const int32_t*>(base + kOffTok);
  rd.blk_start = reinterpret_cast<const int32_t*>(base + kOffStart);
  rd.pos = nullptr;   // positions are looked up from the tables above
  PoolDev pd;
  pd.base = static_cast<uint16_t*>(pool->base);
  pd.num_pages = pool->num_pages;
  pd.bt = pool->block_table;
  pd.max_lp = pool->max_pages_per_agent;
  pd.P = s.page_size;
  pd.p_shift = -1;
  if ((s.page_size & (s.page_size - 1)) == 0) {
    pd.p_shift = 0;
    while ((1 << pd.p_shift) < s.page_size) ++pd.p_shift;
  }
  float* dev = reinterpret_cast<float*>(base + kOffDev);
  *k_out = k;
  cudaError_t e = launch_deviation(g, rd, pd, check_layer, static_cast<const uint16_t*>(k_fresh),
                                   dev, err, st);
  if (e == cudaSuccess) e = launch_select(dev, N, rd.S, k, sel, st);
  if (e != cudaSuccess) return TD_ERR_CUDA;
  if (err_bits_out) {
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return TD_ERR_CUDA;
    *err_bits_out = bits;
    for (int code = 1; code < 32; ++code)
      if (bits & (1u << code)) return static_cast<td_status>(code);
  }
  return TD_OK;
}
