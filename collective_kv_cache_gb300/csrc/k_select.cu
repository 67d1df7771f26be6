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
// devsel_kernel (td_check_select) fuses both: many CTAs per agent compute deviations and a
// shared first-digit histogram; the agent's last CTA finishes the selection.
// select_kernel is the one-CTA-per-agent select over deviations already in memory (the
// group-wide variant and the allocation-free entry point use it).
#include "td_device.cuh"

namespace td {

// ---- Fused deviation and selection (td_check_select).
// A CTA takes kSelTok consecutive tokens of one agent (grid: agent-major, so an agent's
// CTAs are scheduled together and its tail can start while later agents still stream).
// Its threads first find the pool row of every token (the agent's offsets and the block
// starts staged in shared memory, so the block table is the only dependent global load),
// then each warp computes the deviations of its tokens with their loads in flight
// together. Each CTA adds its keys to the agent's histogram of the first 12-bit digit
// (warp-aggregated atomics); the CTA that finishes last for its agent (a self-resetting
// counter; no CTA waits) resolves the other 20 bits in two 10-bit passes over the agent's
// keys and writes the ordered selection, then clears the histogram for the next call.
constexpr int kSelTok = 64;         // tokens per CTA
constexpr int kSelThreads = 256;
constexpr int kSelTabM = 256;       // rounds with at most this many blocks stage tables
constexpr int kSelBins1 = kSelHistBins;  // first digit: key bits 31..20
constexpr int kSelBins2 = 1024;     // second and third digits: bits 19..10 and 9..0
constexpr int kSelKeysReg = 16;     // keys a tail thread keeps in registers

struct SelArgs {
  Geom g;
  RoundDev rd;
  PoolDev pool;
  int check_layer;
  const uint16_t* kf;   // [N][S][E] recomputed K at the check layer
  float* dev;           // [N][S]
  int k;
  int32_t* sel;         // [N][k]
  uint32_t* hist;       // [N][kSelBins1], zero between calls; nullptr: deviations only
  int* done;            // [N] CTAs finished per agent, zero between calls
  uint32_t* err;
};

// Exclusive prefix over the CTA's kSelThreads threads in thread order; *total gets the sum.
template <typename T>
__device__ __forceinline__ T block_excl_scan(T x, T* s_warp, T* total) {
  constexpr int kWarps = kSelThreads / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  T incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  T w[kWarps];
#pragma unroll
  for (int q = 0; q < kWarps; ++q) w[q] = s_warp[q];
  T before = 0, tot = 0;
#pragma unroll
  for (int q = 0; q < kWarps; ++q) {
    before += q < wid ? w[q] : T(0);
    tot += w[q];
  }
  *total = tot;
  return before + incl - x;
}

// One radix digit over a histogram laid out highest bin first across the threads: thread
// r holds the counts h[0..kPer) of bins top - kPer*r - 1 - q. Finds the bin holding the
// need-th largest key (need >= 1), how many keys of that bin are still needed and how many
// keys the bin holds.
template <int kPer>
__device__ __forceinline__ void find_digit(const uint32_t (&h)[kPer], int top, int need,
                                           unsigned* s_warp, int* s_digit, int* s_need,
                                           int* s_count) {
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
    *s_digit = digit;
    *s_need = left;
    *s_count = count;
  }
  __syncthreads();
}

// The last CTA of agent i: the k largest keys (ties to the lower token), ascending.
// s_h2, s_h3: kSelBins2 counters each in shared memory.
__device__ void select_tail(const uint32_t* __restrict__ keys, int S, int k,
                            uint32_t* __restrict__ hist_i, int32_t* __restrict__ out,
                            uint32_t* s_h2, uint32_t* s_h3) {
  __shared__ unsigned s_warp[kSelThreads / 32];
  __shared__ unsigned long long s_warp64[kSelThreads / 32];
  __shared__ int s_d1, s_d2, s_d3, s_need1, s_need2, s_need3, s_cnt1, s_cnt2, s_cnt3;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int b = tid; b < kSelBins2; b += nthr) {
    s_h2[b] = 0u;
    s_h3[b] = 0u;
  }
  // the thread's contiguous range of tokens; its keys and its 16 first-digit bins are
  // loaded together
  const int per = (S + nthr - 1) / nthr;
  const int r0 = min(S, tid * per), r1 = min(S, r0 + per);
  const bool cached = per <= kSelKeysReg;
  uint32_t kr[kSelKeysReg];
  // every load is issued before any is used (indices clamped into the agent's span)
  auto load_keys = [&](int c0) {
#pragma unroll
    for (int q = 0; q < kSelKeysReg; ++q) kr[q] = __ldcg(keys + min(r0 + c0 + q, S - 1));
#pragma unroll
    for (int q = 0; q < kSelKeysReg; ++q) kr[q] = r0 + c0 + q < r1 ? kr[q] : 0u;
  };
  if (cached) load_keys(0);
  constexpr int kPer1 = kSelBins1 / kSelThreads;   // 16
  uint32_t h1[kPer1];
  uint4* hp = reinterpret_cast<uint4*>(hist_i + kSelBins1 - kPer1 * (tid + 1));
  {
    uint4 v[kPer1 / 4];
#pragma unroll
    for (int q = 0; q < kPer1 / 4; ++q) v[q] = __ldcg(hp + q);
#pragma unroll
    for (int q = 0; q < kPer1 / 4; ++q) {   // bins from the highest down
      h1[kPer1 - 1 - 4 * q] = v[q].x;
      h1[kPer1 - 2 - 4 * q] = v[q].y;
      h1[kPer1 - 3 - 4 * q] = v[q].z;
      h1[kPer1 - 4 - 4 * q] = v[q].w;
    }
  }
  // each pass visits the thread's keys in token order
  auto for_keys = [&](auto&& fn) {
    for (int c0 = 0; c0 < per; c0 += kSelKeysReg) {
      if (!cached) load_keys(c0);
#pragma unroll
      for (int q = 0; q < kSelKeysReg; ++q)
        if (r0 + c0 + q < r1) fn(kr[q], r0 + c0 + q);
    }
  };
  // digit 1 (bits 31..20)
  find_digit<kPer1>(h1, kSelBins1, k, s_warp, &s_d1, &s_need1, &s_cnt1);
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);   // the counts are consumed: clear them
#pragma unroll                                     // for the next call
    for (int q = 0; q < kPer1 / 4; ++q) __stcg(hp + q, z);
  }
  const unsigned d1 = static_cast<unsigned>(s_d1);
  // The selection is every key above T, and of the keys equal to T the need_eq with the
  // lowest tokens. When the threshold's bin is taken whole, T is the largest key below the
  // bin (need_eq = 0) and the remaining digits are not needed.
  int64_t T = (static_cast<int64_t>(d1) << 20) - 1;
  int need_eq = 0;
  constexpr int kPer2 = kSelBins2 / kSelThreads;   // 4
  if (s_need1 != s_cnt1) {
    // digit 2 (bits 19..10) among the keys of bin d1
    for_keys([&](uint32_t key, int) {
      if ((key >> 20) == d1) atomicAdd(&s_h2[(key >> 10) & 1023u], 1u);
    });
    __syncthreads();
    uint32_t h2[kPer2];
#pragma unroll
    for (int q = 0; q < kPer2; ++q) h2[q] = s_h2[kSelBins2 - 1 - kPer2 * tid - q];
    find_digit<kPer2>(h2, kSelBins2, s_need1, s_warp, &s_d2, &s_need2, &s_cnt2);
    const unsigned p2 = (d1 << 10) | static_cast<unsigned>(s_d2);
    T = (static_cast<int64_t>(p2) << 10) - 1;
    if (s_need2 != s_cnt2) {
      // digit 3 (bits 9..0) among the keys of bin (d1, d2)
      for_keys([&](uint32_t key, int) {
        if ((key >> 10) == p2) atomicAdd(&s_h3[key & 1023u], 1u);
      });
      __syncthreads();
      uint32_t h3[kPer2];
#pragma unroll
      for (int q = 0; q < kPer2; ++q) h3[q] = s_h3[kSelBins2 - 1 - kPer2 * tid - q];
      find_digit<kPer2>(h3, kSelBins2, s_need2, s_warp, &s_d3, &s_need3, &s_cnt3);
      T = (static_cast<int64_t>(p2) << 10) | s_d3;   // the k-th largest key itself
      need_eq = s_need3;
    }
  }
  unsigned long long cnt = 0;
  for_keys([&](uint32_t key, int) {
    const int64_t kk = key;
    cnt += kk > T ? (1ull << 32) : (kk == T ? 1ull : 0ull);
  });
  unsigned long long tot;
  const unsigned long long excl = block_excl_scan<unsigned long long>(cnt, s_warp64, &tot);
  int eq_seen = static_cast<int>(excl & 0xFFFFFFFFull);
  int pos = static_cast<int>(excl >> 32) + min(eq_seen, need_eq);
  for_keys([&](uint32_t key, int t) {
    const int64_t kk = key;
    if (kk > T) {
      if (pos < k) out[pos] = t;
      ++pos;
    } else if (kk == T) {
      if (eq_seen < need_eq) {
        if (pos < k) out[pos] = t;
        ++pos;
      }
      ++eq_seen;
    }
  });
}

// Tokens in flight per warp: the 16-byte vectors of kDepth tokens' two rows (8 KiB a warp).
template <int kVec>
__host__ __device__ constexpr int sel_depth() { return 8 / kVec; }
template <int kVec>
__host__ __device__ constexpr size_t sel_ring_bytes() {
  return static_cast<size_t>(kSelThreads / 32) * sel_depth<kVec>() * 2 * kVec * 32 * sizeof(uint4);
}

template <int kVec>
__global__ void __launch_bounds__(kSelThreads, 3) devsel_kernel(SelArgs a) {
  constexpr int kWarps = kSelThreads / 32;
  constexpr int kPerWarp = kSelTok / kWarps;   // tokens a warp computes: wid + kWarps * q
  constexpr int kDepth = sel_depth<kVec>();
  static_assert(kPerWarp % kDepth == 0, "the ring turns a whole number of times");
  __shared__ int64_t s_row[kSelTok];
  __shared__ uint32_t s_key[kSelTok];
  __shared__ int32_t s_off[kSelTabM], s_bst[kSelTabM];
  __shared__ int s_last;
  extern __shared__ uint4 s_ring[];   // [warp][kDepth][fresh, reused][kVec][lane]
  const int S = a.rd.S, M = a.rd.M;
  const int C = (S + kSelTok - 1) / kSelTok;
  const int i = static_cast<int>(blockIdx.x / C);
  const int t0 = static_cast<int>(blockIdx.x - static_cast<unsigned>(i) * C) * kSelTok;
  const int nt = min(kSelTok, S - t0);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = a.g.E >> 3;                   // 16-byte vectors of a row
  uint4* ring = s_ring + static_cast<size_t>(wid) * kDepth * 2 * kVec * 32;
  // lane l copies, and later reads, only the vectors l, l + 32, ... of a row; the rows are
  // read once, so they go first when L2 needs room
  const uint64_t policy = l2_evict_first();
  auto copy_row = [&](int slot, int which, const uint16_t* row) {
#pragma unroll
    for (int r = 0; r < kVec; ++r)
      if (lane + 32 * r < nv)
        cp_async16_hint(ring + ((slot * 2 + which) * kVec + r) * 32 + lane,
                        row + (lane + 32 * r) * 8, policy);
  };
  auto fresh_row = [&](int x) {
    return a.kf + (static_cast<int64_t>(i) * S + t0 + x) * a.g.E;
  };
  pdl_wait();
  // the recomputed rows of the warp's first tokens need no table: in flight at once
#pragma unroll
  for (int u = 0; u < kDepth; ++u)
    if (wid + kWarps * u < nt) copy_row(u, 0, fresh_row(wid + kWarps * u));
  cp_async_commit();
  // pool row (in rows of E elements) of each token at the check layer, -1 if unmapped
  const bool staged = M <= kSelTabM;
  if (staged) {
    for (int j = threadIdx.x; j < M; j += blockDim.x) {
      s_off[j] = __ldg(a.rd.off + i * M + j);
      s_bst[j] = __ldg(a.rd.blk_start + j);
    }
    __syncthreads();
  }
  if (threadIdx.x < nt) {
    const int t = t0 + threadIdx.x;
    int o, b0;
    if (staged) {
      int lo = 0, hi = M - 1;   // the last block starting at or before t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_bst[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      o = s_off[lo];
      b0 = s_bst[lo];
    } else {
      const int j = __ldg(a.rd.tok_block + t);
      o = __ldg(a.rd.off + i * M + j);
      b0 = __ldg(a.rd.blk_start + j);
    }
    s_row[threadIdx.x] = pool_row_index(a.pool, i, a.check_layer, 0, o + t - b0, a.err);
  }
  __syncthreads();
  auto reused_row = [&](int x) { return a.pool.base + s_row[x] * a.g.E; };
  // then their reused rows, one group per token: groups complete in order, so token q is
  // ready when at most kDepth - 1 groups are pending
#pragma unroll
  for (int u = 0; u < kDepth; ++u) {
    const int x = wid + kWarps * u;
    if (x < nt && s_row[x] >= 0) copy_row(u, 1, reused_row(x));
    cp_async_commit();
  }
  // deviations: lane l adds (a-b)^2 over the vectors l, l+32, ... of the token's row in
  // ascending element order (fma), then the warp adds its lanes with an xor tree
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int q0 = 0; q0 < kPerWarp; q0 += kDepth) {
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
      const int x = wid + kWarps * (q0 + u);
      cp_async_wait<kDepth - 1>();
      if (x < nt) {                           // uniform across the warp
        const bool mapped = s_row[x] >= 0;
        float acc = 0.0f;
#pragma unroll
        for (int r = 0; r < kVec; ++r) {
          if (lane + 32 * r < nv) {
            float fx[8], rx[8];
            unpack8(ring[((u * 2 + 0) * kVec + r) * 32 + lane], fx);
            unpack8(mapped ? ring[((u * 2 + 1) * kVec + r) * 32 + lane] : z, rx);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float d = __fsub_rn(fx[q], rx[q]);
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
          a.dev[static_cast<int64_t>(i) * S + t0 + x] = acc;
          s_key[x] = __float_as_uint(acc);
        }
      }
      // this thread's cells of the slot are consumed: refill it with token q0 + u + kDepth
      const int xn = x + kWarps * kDepth;
      if (q0 + u + kDepth < kPerWarp && xn < nt) {
        copy_row(u, 0, fresh_row(xn));
        if (s_row[xn] >= 0) copy_row(u, 1, reused_row(xn));
      }
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
  if (!a.hist || a.k <= 0) return;
  __syncthreads();
  // the CTA's keys into the agent's first-digit histogram, one atomic per distinct digit
  // of a warp
  if (threadIdx.x < kSelTok) {
    const bool live = static_cast<int>(threadIdx.x) < nt;
    const unsigned d = live ? (s_key[threadIdx.x] >> 20) : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
    if (live && lane == __ffs(peers) - 1)
      atomicAdd(a.hist + static_cast<int64_t>(i) * kSelBins1 + d, __popc(peers));
  }
  __syncthreads();
  pdl_trigger();   // the next kernel may be scheduled; it waits for this grid to finish
  // thread 0 publishes the CTA's deviations and counts (release after the barrier) and
  // learns whether it is the agent's last CTA
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(a.done + i, 1) == C - 1;
    if (last) {
      __threadfence();
      a.done[i] = 0;                          // ready for the next call
    }
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;                        // uniform across the CTA
  // the ring is drained: its first 8 KiB hold the tail's histograms
  static_assert(sel_ring_bytes<kVec>() >= 2 * kSelBins2 * sizeof(uint32_t), "tail histograms");
  uint32_t* s_h = reinterpret_cast<uint32_t*>(s_ring);
  select_tail(reinterpret_cast<const uint32_t*>(a.dev + static_cast<int64_t>(i) * S), S, a.k,
              a.hist + static_cast<int64_t>(i) * kSelBins1, a.sel + static_cast<int64_t>(i) * a.k,
              s_h, s_h + kSelBins2);
}

template <int kVec>
static cudaError_t launch_devsel_t(const SelArgs& a, cudaStream_t st) {
  const int64_t C = (a.rd.S + kSelTok - 1) / kSelTok;
  const int64_t blocks = C * a.rd.N;
  if (blocks == 0) return cudaSuccess;
  // the ring is beyond the default shared-memory window: opt in once per device
  static int opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev]) {
    e = cudaFuncSetAttribute(devsel_kernel<kVec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sel_ring_bytes<kVec>()));
    if (e != cudaSuccess) return e;
    opted_in[dev] = 1;
  }
  return launch_after(devsel_kernel<kVec>, static_cast<unsigned>(blocks), kSelThreads,
                      sel_ring_bytes<kVec>(), st, a);
}

// ---- The same stage with one thread-block cluster per agent (rounds of at most
// kClMaxTok * 16 shared tokens). The agent's CTAs keep their deviations in shared memory
// and add them to one first-digit histogram in the leader CTA's shared memory (distributed
// shared memory); a hardware cluster barrier replaces the counter, and the leader reads
// the other CTAs' keys from their shared memory instead of from L2.
constexpr int kClMaxTok = 1024;       // tokens per CTA
constexpr int kClMaxSize = 16;        // CTAs per cluster (non-portable above 8)
constexpr int kClBins1 = 2048;        // digits: bits 31..21, 20..10, 9..0
constexpr int kClBins2 = 2048;
constexpr int kClBins3 = 1024;

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `p` (a shared-memory variable) in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, unsigned rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// The generic address of `p` (a shared-memory variable) in CTA `rank`: plain loads through
// it read that CTA's shared memory.
__device__ __forceinline__ const uint32_t* dsmem_ptr(const uint32_t* p, unsigned rank) {
  uint64_t r;
  asm("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(p), "r"(rank));
  return reinterpret_cast<const uint32_t*>(r);
}

// The leader's part: the k largest keys of the agent (ties to the lower token), ascending.
// s_all holds the agent's S keys (token order) and s_h1 its first-digit histogram, both in
// the leader's shared memory.
__device__ void select_tail_cluster(const uint32_t* s_all, int S, int k, const uint32_t* s_h1,
                                    int32_t* __restrict__ out, uint32_t* s_h2, uint32_t* s_h3) {
  __shared__ unsigned s_warp[kSelThreads / 32];
  __shared__ unsigned long long s_warp64[kSelThreads / 32];
  __shared__ int s_d1, s_d2, s_d3, s_need1, s_need2, s_need3, s_cnt1, s_cnt2, s_cnt3;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int b = tid; b < kClBins2; b += nthr) s_h2[b] = 0u;
  for (int b = tid; b < kClBins3; b += nthr) s_h3[b] = 0u;
  const int per = (S + nthr - 1) / nthr;
  const int r0 = min(S, tid * per), r1 = min(S, r0 + per);
  auto for_keys = [&](auto&& fn) {
    for (int t = r0; t < r1; ++t) fn(s_all[t], t);
  };
  constexpr int kPer1 = kClBins1 / kSelThreads;    // 8
  uint32_t h1[kPer1];
#pragma unroll
  for (int q = 0; q < kPer1; ++q) h1[q] = s_h1[kClBins1 - 1 - kPer1 * tid - q];
  find_digit<kPer1>(h1, kClBins1, k, s_warp, &s_d1, &s_need1, &s_cnt1);
  const unsigned d1 = static_cast<unsigned>(s_d1);
  int64_t T = (static_cast<int64_t>(d1) << 21) - 1;
  int need_eq = 0;
  if (s_need1 != s_cnt1) {
    for_keys([&](uint32_t key, int) {
      if ((key >> 21) == d1) atomicAdd(&s_h2[(key >> 10) & 2047u], 1u);
    });
    __syncthreads();
    constexpr int kPer2 = kClBins2 / kSelThreads;  // 8
    uint32_t h2[kPer2];
#pragma unroll
    for (int q = 0; q < kPer2; ++q) h2[q] = s_h2[kClBins2 - 1 - kPer2 * tid - q];
    find_digit<kPer2>(h2, kClBins2, s_need1, s_warp, &s_d2, &s_need2, &s_cnt2);
    const unsigned p2 = (d1 << 11) | static_cast<unsigned>(s_d2);
    T = (static_cast<int64_t>(p2) << 10) - 1;
    if (s_need2 != s_cnt2) {
      for_keys([&](uint32_t key, int) {
        if ((key >> 10) == p2) atomicAdd(&s_h3[key & 1023u], 1u);
      });
      __syncthreads();
      constexpr int kPer3 = kClBins3 / kSelThreads;  // 4
      uint32_t h3[kPer3];
#pragma unroll
      for (int q = 0; q < kPer3; ++q) h3[q] = s_h3[kClBins3 - 1 - kPer3 * tid - q];
      find_digit<kPer3>(h3, kClBins3, s_need2, s_warp, &s_d3, &s_need3, &s_cnt3);
      T = (static_cast<int64_t>(p2) << 10) | s_d3;
      need_eq = s_need3;
    }
  }
  unsigned long long cnt = 0;
  for_keys([&](uint32_t key, int) {
    const int64_t kk = key;
    cnt += kk > T ? (1ull << 32) : (kk == T ? 1ull : 0ull);
  });
  unsigned long long tot;
  const unsigned long long excl = block_excl_scan<unsigned long long>(cnt, s_warp64, &tot);
  int eq_seen = static_cast<int>(excl & 0xFFFFFFFFull);
  int pos = static_cast<int>(excl >> 32) + min(eq_seen, need_eq);
  for_keys([&](uint32_t key, int t) {
    const int64_t kk = key;
    if (kk > T) {
      if (pos < k) out[pos] = t;
      ++pos;
    } else if (kk == T) {
      if (eq_seen < need_eq) {
        if (pos < k) out[pos] = t;
        ++pos;
      }
      ++eq_seen;
    }
  });
}

// Shared memory of the cluster kernel beyond its static part: the ring, then the leader's
// copy of the agent's keys.
template <int kVec>
__host__ __device__ constexpr size_t cl_keys_offset() { return sel_ring_bytes<kVec>(); }
template <int kVec>
__host__ __device__ constexpr size_t cl_dynamic_bytes(int S) {
  return cl_keys_offset<kVec>() + ((static_cast<size_t>(S) * 4 + 15) & ~size_t(15));
}

// grid: N clusters of C CTAs; CTA r of agent i takes tokens [r * tpc, min(S, (r+1) * tpc)).
// Every thread of every CTA passes the same cluster barrier phases: (0) every CTA of the
// cluster runs and its histogram is zero, (A) keys and counts are in the leader's shared
// memory; then every CTA but the leader exits.
template <int kVec>
__global__ void __launch_bounds__(kSelThreads, 2) devsel_cluster_kernel(SelArgs a, int C,
                                                                        int tpc) {
  constexpr int kWarps = kSelThreads / 32;
  constexpr int kDepth = sel_depth<kVec>();
  __shared__ int64_t s_row[kClMaxTok];
  __shared__ uint32_t s_key[kClMaxTok];
  __shared__ uint32_t s_hist[kClBins1];
  __shared__ int32_t s_off[kSelTabM], s_bst[kSelTabM];
  extern __shared__ uint4 s_ring[];   // [warp][kDepth][fresh, reused][kVec][lane], then keys
  uint32_t* s_all = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(s_ring) +
                                                cl_keys_offset<kVec>());
  const int S = a.rd.S, M = a.rd.M;
  const unsigned rank = cluster_rank();
  const int i = static_cast<int>(blockIdx.x) / C;
  const int t0 = static_cast<int>(rank) * tpc;
  const int ntok = max(0, min(tpc, S - t0));
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = a.g.E >> 3;
  const int nq = ntok > wid ? (ntok - wid + kWarps - 1) / kWarps : 0;   // this warp's tokens
  uint4* ring = s_ring + static_cast<size_t>(wid) * kDepth * 2 * kVec * 32;
  const uint64_t policy = l2_evict_first();
  auto copy_row = [&](int slot, int which, const uint16_t* row) {
#pragma unroll
    for (int r = 0; r < kVec; ++r)
      if (lane + 32 * r < nv)
        cp_async16_hint(ring + ((slot * 2 + which) * kVec + r) * 32 + lane,
                        row + (lane + 32 * r) * 8, policy);
  };
  auto fresh_row = [&](int x) {
    return a.kf + (static_cast<int64_t>(i) * S + t0 + x) * a.g.E;
  };
  for (int b = threadIdx.x; b < kClBins1; b += blockDim.x) s_hist[b] = 0u;
  cluster_arrive_relaxed();                       // (0) this CTA runs; its histogram is zero
  pdl_wait();
#pragma unroll
  for (int u = 0; u < kDepth; ++u)
    if (u < nq) copy_row(u, 0, fresh_row(wid + kWarps * u));
  cp_async_commit();
  const bool staged = M <= kSelTabM;
  if (staged) {
    for (int j = threadIdx.x; j < M; j += blockDim.x) {
      s_off[j] = __ldg(a.rd.off + i * M + j);
      s_bst[j] = __ldg(a.rd.blk_start + j);
    }
    __syncthreads();
  }
  for (int x = threadIdx.x; x < ntok; x += blockDim.x) {
    const int t = t0 + x;
    int o, b0;
    if (staged) {
      int lo = 0, hi = M - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_bst[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      o = s_off[lo];
      b0 = s_bst[lo];
    } else {
      const int j = __ldg(a.rd.tok_block + t);
      o = __ldg(a.rd.off + i * M + j);
      b0 = __ldg(a.rd.blk_start + j);
    }
    s_row[x] = pool_row_index(a.pool, i, a.check_layer, 0, o + t - b0, a.err);
  }
  __syncthreads();
  auto reused_row = [&](int x) { return a.pool.base + s_row[x] * a.g.E; };
#pragma unroll
  for (int u = 0; u < kDepth; ++u) {
    const int x = wid + kWarps * u;
    if (u < nq && s_row[x] >= 0) copy_row(u, 1, reused_row(x));
    cp_async_commit();
  }
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int q0 = 0; q0 < nq; q0 += kDepth) {
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
      const int q = q0 + u;
      const int x = wid + kWarps * q;
      cp_async_wait<kDepth - 1>();
      if (q < nq) {                               // uniform across the warp
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
            acc = 0.0f;
          } else if (!isfinite(acc)) {
            atomicOr(a.err, err_bit(TD_ERR_NONFINITE));
          }
          a.dev[static_cast<int64_t>(i) * S + t0 + x] = acc;
          s_key[x] = __float_as_uint(acc);
        }
      }
      const int qn = q + kDepth;
      if (qn < nq) {
        const int xn = wid + kWarps * qn;
        copy_row(u, 0, fresh_row(xn));
        if (s_row[xn] >= 0) copy_row(u, 1, reused_row(xn));
      }
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  cluster_wait();                                 // (0) every CTA of the cluster runs
  // the CTA's keys into the leader's copy (stores that do not wait) and into its histogram
  // (one atomic per distinct digit of a warp)
  uint32_t* lead_all = const_cast<uint32_t*>(dsmem_ptr(s_all, 0u)) + t0;
  const uint32_t lead_hist = dsmem_addr(s_hist, 0u);
  for (int x0 = 0; x0 < ntok; x0 += blockDim.x) {
    const int x = x0 + threadIdx.x;
    const bool live = x < ntok;
    const uint32_t key = live ? s_key[x] : 0u;
    if (live) lead_all[x] = key;
    const unsigned d = live ? (key >> 21) : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
    if (live && lane == __ffs(peers) - 1) dsmem_add(lead_hist + 4u * d, __popc(peers));
  }
  pdl_trigger();   // the next kernel may be scheduled; it waits for this grid to finish
  cluster_arrive();                               // (A) keys and counts in place (release)
  cluster_wait();
  if (rank != 0) return;
  uint32_t* s_h = reinterpret_cast<uint32_t*>(s_ring);   // the ring is drained
  select_tail_cluster(s_all, S, a.k, s_hist, a.sel + static_cast<int64_t>(i) * a.k, s_h,
                      s_h + kClBins2);
}

template <int kVec>
static cudaError_t launch_devsel_cluster_t(const SelArgs& a, int C, int tpc, cudaStream_t st) {
  static int ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev]) {
    if ((e = cudaFuncSetAttribute(devsel_cluster_kernel<kVec>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(cl_dynamic_bytes<kVec>(kClMaxTok * kClMaxSize)))) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(devsel_cluster_kernel<kVec>,
                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
      return e;
    ready[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C) * static_cast<unsigned>(a.rd.N));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = cl_dynamic_bytes<kVec>(a.rd.S);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, devsel_cluster_kernel<kVec>, a, C, tpc);
}

// Cluster size for a round: up to 16 CTAs of at least 64 tokens; 0 when the round is too
// large for the cluster kernel.
static int cluster_size_for(int S) {
  const int C = min(kClMaxSize, (S + kSelTok - 1) / kSelTok);
  if (C < 1 || (S + C - 1) / C > kClMaxTok) return 0;
  return C;
}

static cudaError_t launch_devsel_cluster(const SelArgs& a, int C, cudaStream_t st) {
  const int tpc = (a.rd.S + C - 1) / C;
  const int nv = a.g.E >> 3;
  if (nv <= 32) return launch_devsel_cluster_t<1>(a, C, tpc, st);
  if (nv <= 64) return launch_devsel_cluster_t<2>(a, C, tpc, st);
  if (nv <= 128) return launch_devsel_cluster_t<4>(a, C, tpc, st);
  return launch_devsel_cluster_t<8>(a, C, tpc, st);
}

static cudaError_t launch_devsel(const SelArgs& a, cudaStream_t st) {
  const int nv = a.g.E >> 3;
  if (nv <= 32) return launch_devsel_t<1>(a, st);
  if (nv <= 64) return launch_devsel_t<2>(a, st);
  if (nv <= 128) return launch_devsel_t<4>(a, st);
  return launch_devsel_t<8>(a, st);
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
  SelArgs a{g, rd, pool, check_layer, k_fresh, dev, 0, nullptr, nullptr, nullptr, err};
  return launch_devsel(a, st);
}

cudaError_t launch_select(const float* dev, int N, int S, int k, int32_t* sel,
                          cudaStream_t st) {
  if (k <= 0 || N <= 0) return cudaSuccess;
  return launch_after(select_kernel, static_cast<unsigned>(N), 1024, 0, st, dev, S, k, sel);
}

cudaError_t launch_check_select(const Geom& g, const RoundDev& rd, const PoolDev& pool,
                                int check_layer, const uint16_t* k_fresh, float* dev, int k,
                                int32_t* sel, uint32_t* hist, int* done, uint32_t* err,
                                cudaStream_t st) {
  SelArgs a{g, rd, pool, check_layer, k_fresh, dev, k, sel, hist, done, err};
  const int C = k > 0 ? cluster_size_for(rd.S) : 0;
  if (C > 0) return launch_devsel_cluster(a, C, st);
  return launch_devsel(a, st);
}

}  // namespace td
