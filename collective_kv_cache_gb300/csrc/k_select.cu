// k_select.cu - stage 2: key deviation at the check layer and per-agent top-k
// (TokenDance review [R], Summary Method (2): one key-difference analysis for the whole
// group at the check layer; its important positions are reused by all later layers).
//
// The deviation of (agent, token) is the squared L2 distance between the recomputed K and
// the reused K in the agent's pages, in a fixed order that is part of the definition (the
// selection is compared bit for bit): lane l of a warp takes the 16-byte vectors l, l+32,
// ... of the row and adds (a-b)^2 with fma in ascending element order, then the warp adds
// its 32 partial sums with an xor butterfly (16, 8, 4, 2, 1).
// The selection is a radix select on the float bits of the deviations (non-negative, so
// the bits order like the values): it finds the k-th largest value T and takes every
// token above T and the lowest-index tokens equal to T, in ascending token order.
//
// Two launches, the second a programmatic dependent launch of the first:
//   dev_kernel   the round's N*S (agent, token) pairs are cut into one equal range per
//                resident CTA (one wave, two CTAs an SM), so every SM moves the same
//                bytes. Each warp takes every eighth token of the range through a ring of
//                12 KiB of shared memory filled by cp.async (16-byte copies, each lane its
//                own cells, refilled the moment a token is consumed). The recomputed rows
//                of the ring's first tokens need no lookup and are in flight first; then
//                the CTA looks up the pool row of each of its tokens (its prompt position
//                from the round's table, then the block table). The deviations go to
//                `dev`; the first 12 bits of each key are counted in the agent's histogram.
//   topk_kernel  one 512-thread CTA per agent: the histogram gives the threshold's first
//                digit, two 10-bit passes over the agent's keys (staged in shared memory)
//                give the rest, and warp ballots in token order write the selection
//                ascending. It clears the histogram for the next call.
#include "td_device.cuh"

namespace td {

// ---- the selection of one agent (one 512-thread CTA)
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelBins2 = 1024;        // second and third digits: bits 19..10 and 9..0
constexpr int kSelKeysSmem = 16384;    // keys an agent's selection stages (64 KiB)

// Exclusive prefix over the CTA's kSelThreads threads in thread order; *total gets the sum.
template <typename T>
__device__ __forceinline__ T block_excl_scan(T x, T* s_warp, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  T incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  // every warp scans the warp totals itself: lane q holds the total of warp q
  const T w = lane < kSelWarps ? s_warp[lane] : T(0);
  T wincl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
    if (lane >= o) wincl += y;
  }
  const T before = __shfl_sync(0xFFFFFFFFu, wincl - w, wid);
  *total = __shfl_sync(0xFFFFFFFFu, wincl, kSelWarps - 1);
  __syncthreads();   // s_warp may be rewritten by the next scan
  return before + incl - x;
}

// One radix digit over a histogram laid out highest bin first across the threads: thread
// r holds the counts h[0..kPer) of bins top - kPer*r - 1 - q. Finds the bin holding the
// need-th largest key (need >= 1): s_res = {the bin, how many of its keys are still
// needed, how many keys it holds}.
template <int kPer>
__device__ __forceinline__ void find_digit(const uint32_t (&h)[kPer], int top, int need,
                                           unsigned* s_warp, int* s_res) {
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) local += h[q];
  unsigned tot;
  const unsigned excl = block_excl_scan<unsigned>(local, s_warp, &tot);
  if (excl < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= excl + local) {
    unsigned cum = excl;
    int digit = -1, left = 0, count = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (digit < 0) {
        if (cum + h[q] >= static_cast<unsigned>(need)) {
          digit = top - kPer * static_cast<int>(threadIdx.x) - 1 - q;
          left = need - static_cast<int>(cum);
          count = static_cast<int>(h[q]);
        }
        cum += h[q];
      }
    }
    s_res[0] = digit;
    s_res[1] = left;
    s_res[2] = count;
  }
  __syncthreads();
}

// The k largest of one agent's S keys (ties to the lower token), ascending, into out[0..k).
// keys_g: the keys in global memory (written by other CTAs: read through L2). hist_g: their
// first-digit histogram in global memory (read, then cleared), or nullptr to count it here
// in s_h1 (kSelHistBins words). s_keys: kSelKeysSmem words of shared memory, or nullptr
// (the keys are then read from L2 by every pass). s_h: 2 * kSelBins2 words. Every thread of
// the CTA calls it.
__device__ void select_agent(const uint32_t* keys_g, int S, int k, uint32_t* hist_g,
                             int32_t* __restrict__ out, uint32_t* s_keys, uint32_t* s_h1,
                             uint32_t* s_h) {
  __shared__ unsigned s_warp[kSelWarps];
  __shared__ unsigned long long s_warp64[kSelWarps];
  __shared__ int s_d1[3], s_d2[3], s_d3[3];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool staged = s_keys && S <= kSelKeysSmem;
  if (staged) {
    constexpr int kBatch = 4;                         // a thread's loads in flight together
    for (int t0 = 0; t0 < S; t0 += kSelThreads * kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int t = t0 + q * kSelThreads + tid;
        v[q] = t < S ? __ldcg(keys_g + t) : 0u;
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int t = t0 + q * kSelThreads + tid;
        if (t < S) s_keys[t] = v[q];
      }
    }
  }
  auto key_at = [&](int t) { return staged ? s_keys[t] : __ldcg(keys_g + t); };
  constexpr int kPer1 = kSelHistBins / kSelThreads;   // 8
  uint32_t h1[kPer1];
  if (hist_g) {
    uint4* hp = reinterpret_cast<uint4*>(hist_g + kSelHistBins - kPer1 * (tid + 1));
    uint4 v[kPer1 / 4];
#pragma unroll
    for (int q = 0; q < kPer1 / 4; ++q) v[q] = __ldcg(hp + q);
#pragma unroll
    for (int q = 0; q < kPer1 / 4; ++q) {
      __stcg(hp + q, make_uint4(0u, 0u, 0u, 0u));   // consumed: zero for the next call
      h1[kPer1 - 1 - 4 * q] = v[q].x;                // bins from the highest down
      h1[kPer1 - 2 - 4 * q] = v[q].y;
      h1[kPer1 - 3 - 4 * q] = v[q].z;
      h1[kPer1 - 4 - 4 * q] = v[q].w;
    }
    __syncthreads();                                  // the staged keys
  } else {
    for (int b = tid; b < kSelHistBins; b += kSelThreads) s_h1[b] = 0u;
    __syncthreads();                                  // the staged keys, the cleared bins
    for (int t0 = 0; t0 < S; t0 += kSelThreads) {     // uniform trip count
      const int t = t0 + tid;
      const unsigned d = t < S ? (key_at(t) >> 20) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
      if (t < S && lane == __ffs(peers) - 1) atomicAdd(&s_h1[d], static_cast<unsigned>(__popc(peers)));
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPer1; ++q) h1[q] = s_h1[kSelHistBins - 1 - kPer1 * tid - q];
  }
  uint32_t* s_h2 = s_h;
  uint32_t* s_h3 = s_h + kSelBins2;
  for (int b = tid; b < 2 * kSelBins2; b += kSelThreads) s_h[b] = 0u;
  // digit 1 (bits 31..20); find_digit's barriers also order the clearing above
  find_digit<kPer1>(h1, kSelHistBins, k, s_warp, s_d1);
  const unsigned d1 = static_cast<unsigned>(s_d1[0]);
  // The selection is every key above T, and of the keys equal to T the need_eq with the
  // lowest tokens. When the threshold's bin is taken whole, T is the largest key below the
  // bin (need_eq = 0) and the remaining digits are not needed.
  int64_t T = (static_cast<int64_t>(d1) << 20) - 1;
  int need_eq = 0;
  constexpr int kPer2 = kSelBins2 / kSelThreads;   // 2
  if (s_d1[1] != s_d1[2]) {
    // digit 2 (bits 19..10) among the keys of bin d1
    for (int t = tid; t < S; t += kSelThreads) {
      const uint32_t key = key_at(t);
      if ((key >> 20) == d1) atomicAdd(&s_h2[(key >> 10) & 1023u], 1u);
    }
    __syncthreads();
    uint32_t h2[kPer2];
#pragma unroll
    for (int q = 0; q < kPer2; ++q) h2[q] = s_h2[kSelBins2 - 1 - kPer2 * tid - q];
    find_digit<kPer2>(h2, kSelBins2, s_d1[1], s_warp, s_d2);
    const unsigned p2 = (d1 << 10) | static_cast<unsigned>(s_d2[0]);
    T = (static_cast<int64_t>(p2) << 10) - 1;
    if (s_d2[1] != s_d2[2]) {
      // digit 3 (bits 9..0) among the keys of bin (d1, d2)
      for (int t = tid; t < S; t += kSelThreads) {
        const uint32_t key = key_at(t);
        if ((key >> 10) == p2) atomicAdd(&s_h3[key & 1023u], 1u);
      }
      __syncthreads();
      uint32_t h3[kPer2];
#pragma unroll
      for (int q = 0; q < kPer2; ++q) h3[q] = s_h3[kSelBins2 - 1 - kPer2 * tid - q];
      find_digit<kPer2>(h3, kSelBins2, s_d2[1], s_warp, s_d3);
      T = (static_cast<int64_t>(p2) << 10) | s_d3[0];   // the k-th largest key itself
      need_eq = s_d3[1];
    }
  }
  // the output: warp w walks the tokens [w*cw, (w+1)*cw), 32 at a time in token order;
  // ballots of (above T) and (equal to T) give each taken token its place
  const int cw = ((S + kSelWarps - 1) / kSelWarps + 31) & ~31;
  const int w0 = min(S, wid * cw), w1 = min(S, w0 + cw);
  unsigned n_gt = 0, n_eq = 0;
  for (int b = w0; b < w1; b += 32) {
    const int t = b + lane;
    const int64_t kk = t < w1 ? static_cast<int64_t>(key_at(t)) : -1;
    n_gt += __popc(__ballot_sync(0xFFFFFFFFu, kk > T));
    n_eq += __popc(__ballot_sync(0xFFFFFFFFu, kk == T));
  }
  unsigned long long tot;
  const unsigned long long mine = (static_cast<unsigned long long>(n_gt) << 32) | n_eq;
  const unsigned long long excl =
      block_excl_scan<unsigned long long>(lane == 0 ? mine : 0ull, s_warp64, &tot);
  const unsigned long long wex = __shfl_sync(0xFFFFFFFFu, excl, 0);
  int eq_seen = static_cast<int>(wex & 0xFFFFFFFFull);
  int pos = static_cast<int>(wex >> 32) + min(eq_seen, need_eq);
  const unsigned below = (1u << lane) - 1u;
  for (int b = w0; b < w1; b += 32) {
    const int t = b + lane;
    const int64_t kk = t < w1 ? static_cast<int64_t>(key_at(t)) : -1;
    const unsigned gt = __ballot_sync(0xFFFFFFFFu, kk > T);
    const unsigned eq = __ballot_sync(0xFFFFFFFFu, kk == T);
    // the equal keys still wanted: the first need_eq - eq_seen of this group's
    const int want = max(0, min(32, need_eq - eq_seen));
    const bool take_eq = (eq >> lane) & 1u && __popc(eq & below) < want;
    const unsigned taken = gt | __ballot_sync(0xFFFFFFFFu, take_eq);
    if ((taken >> lane) & 1u) {
      const int p = pos + __popc(taken & below);
      if (p < k) out[p] = t;
    }
    pos += __popc(taken);
    eq_seen += __popc(eq);
  }
}

// ---- dev_kernel
constexpr int kDevThreads = 256;
constexpr int kDevWarps = kDevThreads / 32;
constexpr int kDevCtasPerSm = 2;
constexpr int kDevMaxTok = 1024;          // (agent, token) pairs per CTA at most
constexpr int kDevWarpRing = 12 * 1024;   // bytes of rows a warp has in flight

struct DevArgs {
  Geom g;
  RoundDev rd;
  PoolDev pool;
  int check_layer;
  const uint16_t* kf;   // [N][S][E] recomputed K at the check layer
  float* dev;           // [N][S]
  uint32_t* hist;       // [N][kSelHistBins] first-digit counts, zero between calls; nullptr:
                        // not counted
  uint32_t* err;
  int per_cta;          // (agent, token) pairs per CTA
};

// The prompt position of every token of the round (one thread a token).
__global__ void __launch_bounds__(256) positions_kernel(RoundDev rd, int32_t* pos) {
  const int64_t total = static_cast<int64_t>(rd.N) * rd.S;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(g / rd.S);
    const int t = static_cast<int>(g - static_cast<int64_t>(i) * rd.S);
    const int j = rd.tok_block[t];
    pos[g] = rd.off[i * rd.M + j] + t - rd.blk_start[j];
  }
}

cudaError_t launch_positions(const RoundDev& rd, int32_t* pos, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(rd.N) * rd.S;
  const int64_t blocks = (total + 255) / 256;
  positions_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(rd,
                                                                                        pos);
  return cudaGetLastError();
}

// kVec: 16-byte vectors a lane takes of a row (lane l: vectors l, l + 32, ...); kSlots:
// tokens in a warp's ring (both rows of a token in one slot, 12 KiB a warp).
template <int kVec, int kSlots>
__global__ void __launch_bounds__(kDevThreads, kDevCtasPerSm) dev_kernel(DevArgs a) {
  __shared__ int64_t s_row[kDevMaxTok];   // pool row of each token, -1 unmapped
  __shared__ uint32_t s_key[kDevMaxTok];
  extern __shared__ uint4 s_ring[];       // [warp][slot][recomputed, reused][kVec][lane]
  const int S = a.rd.S, M = a.rd.M, E = a.g.E;
  const int64_t total = static_cast<int64_t>(a.rd.N) * S;
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * a.per_cta;
  const int n = static_cast<int>(min(static_cast<int64_t>(a.per_cta), total - g0));
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nv = E >> 3;                      // 16-byte vectors of a row
  const int nq = n > wid ? (n - wid + kDevWarps - 1) / kDevWarps : 0;   // this warp's tokens
  uint4* ring = s_ring + static_cast<size_t>(wid) * kSlots * 2 * kVec * 32;
  const uint64_t policy = l2_evict_first();   // every row is read once
  // lane l copies, and later reads, only its own cells: no barrier, only the group waits
  auto copy_row = [&](int slot, int which, const uint16_t* row) {
#pragma unroll
    for (int r = 0; r < kVec; ++r)
      if (lane + 32 * r < nv)
        cp_async16_hint(ring + ((slot * 2 + which) * kVec + r) * 32 + lane,
                        row + (lane + 32 * r) * 8, policy);
  };
  auto fresh_row = [&](int q) { return a.kf + (g0 + wid + q * kDevWarps) * E; };
  auto reused_row = [&](int q) { return a.pool.base + s_row[wid + q * kDevWarps] * E; };
  pdl_wait();
  // the prompt position of every token of the range first (its loads head the queue), then
  // the recomputed rows of the ring's first tokens (they need no lookup), then the block
  // table at those positions -> the pool rows
  constexpr int kPer = kDevMaxTok / kDevThreads;
  int pos[kPer], ag[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int x = min(tid + q * kDevThreads, n - 1);
    const int64_t g = g0 + x;
    ag[q] = static_cast<int>(g / S);
    if (a.rd.pos) {
      pos[q] = __ldg(a.rd.pos + g);
    } else {
      const int t = static_cast<int>(g - static_cast<int64_t>(ag[q]) * S);
      const int j = __ldg(a.rd.tok_block + t);
      pos[q] = __ldg(a.rd.off + ag[q] * M + j) + t - __ldg(a.rd.blk_start + j);
    }
  }
#pragma unroll
  for (int q = 0; q < kSlots; ++q)
    if (q < nq) copy_row(q, 0, fresh_row(q));
  cp_async_commit();
#pragma unroll
  for (int q = 0; q < kPer; ++q)
    if (tid + q * kDevThreads < n)
      s_row[tid + q * kDevThreads] =
          pool_row_index(a.pool, ag[q], a.check_layer, 0, pos[q], a.err);
  __syncthreads();
  // then their reused rows, one group per token: groups complete in order, so token q has
  // landed when at most kSlots - 1 groups are pending
#pragma unroll
  for (int q = 0; q < kSlots; ++q) {
    if (q < nq && s_row[wid + q * kDevWarps] >= 0) copy_row(q, 1, reused_row(q));
    cp_async_commit();
  }
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int q0 = 0; q0 < nq; q0 += kSlots) {
#pragma unroll
    for (int u = 0; u < kSlots; ++u) {
      const int q = q0 + u;
      cp_async_wait<kSlots - 1>();
      if (q < nq) {                           // uniform across the warp
        const int x = wid + q * kDevWarps;
        const bool mapped = s_row[x] >= 0;
        float acc = 0.0f;
#pragma unroll
        for (int r = 0; r < kVec; ++r) {
          if (lane + 32 * r < nv) {
            float fx[8], rx[8];
            unpack8(ring[((u * 2 + 0) * kVec + r) * 32 + lane], fx);
            unpack8(mapped ? ring[((u * 2 + 1) * kVec + r) * 32 + lane] : z, rx);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float d = __fsub_rn(fx[e], rx[e]);
              acc = __fmaf_rn(d, d, acc);
            }
          }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
          acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
        if (lane == 0) {
          if (!mapped) {
            acc = 0.0f;                       // unmapped: reported, deviation 0
          } else if (!isfinite(acc)) {
            atomicOr(a.err, err_bit(TD_ERR_NONFINITE));
          }
          s_key[x] = __float_as_uint(acc);
        }
      }
      // this lane's cells of the slot are consumed: refill it with token q + kSlots
      const int qn = q + kSlots;
      if (qn < nq) {
        copy_row(u, 0, fresh_row(qn));
        if (s_row[wid + qn * kDevWarps] >= 0) copy_row(u, 1, reused_row(qn));
      }
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  pdl_trigger();   // the top-k may be scheduled; it waits for this grid to finish
  // the range's deviations (coalesced) and its keys into the agents' histograms, one
  // atomic per distinct (agent, first digit) of a warp
  for (int x0 = 0; x0 < n; x0 += kDevThreads) {
    const int x = x0 + tid;
    const bool live = x < n;
    const uint32_t key = live ? s_key[x] : 0u;
    if (live) a.dev[g0 + x] = __uint_as_float(key);
    if (a.hist) {
      const int i = live ? static_cast<int>((g0 + x) / S) : 0;
      const unsigned id = live ? (static_cast<unsigned>(i) << 12) | (key >> 20) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, id);
      if (live && lane == __ffs(peers) - 1)
        atomicAdd(a.hist + static_cast<int64_t>(i) * kSelHistBins + (key >> 20),
                  static_cast<unsigned>(__popc(peers)));
    }
  }
}

template <int kVec, int kSlots>
static cudaError_t launch_dev_t(const DevArgs& a0, cudaStream_t st) {
  constexpr size_t kRing = static_cast<size_t>(kDevWarps) * kSlots * 2 * kVec * 32 * 16;
  static int sms[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sms[dev]) {   // the rings pass the default shared-memory window: opt in once
    int n = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dev_kernel<kVec, kSlots>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kRing))) != cudaSuccess)
      return e;
    sms[dev] = n;
  }
  DevArgs a = a0;
  const int64_t total = static_cast<int64_t>(a.rd.N) * a.rd.S;
  if (total == 0) return cudaSuccess;
  // one equal range per resident CTA (one wave), at most kDevMaxTok pairs each
  const int64_t slots = static_cast<int64_t>(sms[dev]) * kDevCtasPerSm;
  int64_t per = (total + slots - 1) / slots;
  if (per > kDevMaxTok) per = kDevMaxTok;
  a.per_cta = static_cast<int>(per);
  return launch_after(dev_kernel<kVec, kSlots>, static_cast<unsigned>((total + per - 1) / per),
                      kDevThreads, kRing, st, a);
}

static cudaError_t launch_dev(const DevArgs& a, cudaStream_t st) {
  const int nv = a.g.E >> 3;   // ring slots: kDevWarpRing / (2 rows of kVec * 512 bytes)
  if (nv <= 32) return launch_dev_t<1, 12>(a, st);
  if (nv <= 64) return launch_dev_t<2, 6>(a, st);
  if (nv <= 128) return launch_dev_t<4, 3>(a, st);
  return launch_dev_t<8, 2>(a, st);
}

// ---- topk_kernel: one CTA per row of keys already in memory. hist: the rows' first-digit
// histograms (read, then cleared), or nullptr to count them here.
__global__ void __launch_bounds__(kSelThreads)
topk_kernel(const float* __restrict__ dev, int S, int k, int32_t* __restrict__ sel,
            uint32_t* hist) {
  __shared__ uint32_t s_h1[kSelHistBins];
  __shared__ uint32_t s_h[2 * kSelBins2];
  extern __shared__ uint32_t s_keys[];
  pdl_wait();
  const int i = blockIdx.x;
  select_agent(reinterpret_cast<const uint32_t*>(dev) + static_cast<int64_t>(i) * S, S, k,
               hist ? hist + static_cast<int64_t>(i) * kSelHistBins : nullptr,
               sel + static_cast<int64_t>(i) * k, S <= kSelKeysSmem ? s_keys : nullptr, s_h1,
               s_h);
}

static cudaError_t launch_topk(const float* dev, int N, int S, int k, int32_t* sel,
                               uint32_t* hist, cudaStream_t st) {
  if (k <= 0 || N <= 0) return cudaSuccess;
  static int opted[64] = {};
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (!opted[d]) {   // the staged keys pass the default shared-memory window
    if ((e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSelKeysSmem * 4)) != cudaSuccess)
      return e;
    opted[d] = 1;
  }
  const size_t smem = static_cast<size_t>(S < kSelKeysSmem ? S : kSelKeysSmem) * 4;
  return launch_after(topk_kernel, static_cast<unsigned>(N), kSelThreads, smem, st, dev, S, k,
                      sel, hist);
}

cudaError_t launch_deviation(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                             int check_layer, const uint16_t* k_fresh, float* dev,
                             uint32_t* err, cudaStream_t st) {
  const DevArgs a{g, rd, pool, check_layer, k_fresh, dev, nullptr, err, 0};
  return launch_dev(a, st);
}

cudaError_t launch_select(const float* dev, int N, int S, int k, int32_t* sel,
                          cudaStream_t st) {
  return launch_topk(dev, N, S, k, sel, nullptr, st);
}

cudaError_t launch_check_select(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                int check_layer, const uint16_t* k_fresh, float* dev, int k,
                                int32_t* sel, uint32_t* hist, uint32_t* err, cudaStream_t st) {
  const DevArgs a{g, rd, pool, check_layer, k_fresh, dev, k > 0 ? hist : nullptr, err, 0};
  cudaError_t e = launch_dev(a, st);
  if (e != cudaSuccess) return e;
  return launch_topk(dev, rd.N, rd.S, k, sel, hist, st);
}

}  // namespace td
