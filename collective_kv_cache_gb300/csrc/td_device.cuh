// td_device.cuh - device helpers: bf16 packing, the RoPE pair-vector rotation, tile
// geometry and the paged-KV address of a token row.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "td_internal.h"

namespace td {

// ---- bf16 words: a 32-bit word holds two bf16 values, the lower address in the low half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> two bf16, round to nearest even, in one instruction.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* x) {
  x[0] = bf_lo(v.x); x[1] = bf_hi(v.x); x[2] = bf_lo(v.y); x[3] = bf_hi(v.y);
  x[4] = bf_lo(v.z); x[5] = bf_hi(v.z); x[6] = bf_lo(v.w); x[7] = bf_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float* y) {
  return make_uint4(pack_bf2(y[0], y[1]), pack_bf2(y[2], y[3]), pack_bf2(y[4], y[5]),
                    pack_bf2(y[6], y[7]));
}

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld16(const uint16_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void st16(uint16_t* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ bool neq16(const uint4& a, const uint4& b) {
  return ((a.x ^ b.x) | (a.y ^ b.y) | (a.z ^ b.z) | (a.w ^ b.w)) != 0u;
}

// ---- RoPE on one pair-vector: 8 consecutive frequencies f0..f0+7 of one head.
// a holds elements f0..f0+7, b holds f0+D/2..f0+D/2+7; c, s point at cos/sin[f0].
// forward:  y0 = fma(x0, c, -(x1*s)),  y1 = fma(x1, c, x0*s)
// inverse:  y0 = fma(x0, c,  x1*s),    y1 = fma(x1, c, -(x0*s))
// Each cross product is rounded to float before the fma; outputs rounded to bf16.
template <bool kInverse>
__device__ __forceinline__ void rotate_pairs(const uint4& a, const uint4& b, const float* c,
                                             const float* s, uint4& ya, uint4& yb) {
  float x0[8], x1[8], y0[8], y1[8];
  unpack8(a, x0);
  unpack8(b, x1);
  const float4 c0 = __ldg(reinterpret_cast<const float4*>(c));
  const float4 c1 = __ldg(reinterpret_cast<const float4*>(c) + 1);
  const float4 s0 = __ldg(reinterpret_cast<const float4*>(s));
  const float4 s1 = __ldg(reinterpret_cast<const float4*>(s) + 1);
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float x1s = __fmul_rn(x1[q], ss[q]);
    const float x0s = __fmul_rn(x0[q], ss[q]);
    if (kInverse) {
      y0[q] = __fmaf_rn(x0[q], cc[q], x1s);
      y1[q] = __fmaf_rn(x1[q], cc[q], -x0s);
    } else {
      y0[q] = __fmaf_rn(x0[q], cc[q], -x1s);
      y1[q] = __fmaf_rn(x1[q], cc[q], x0s);
    }
  }
  ya = pack8(y0);
  yb = pack8(y1);
}

// ---- Tile geometry: a tile is (layer, kTile = 16 canonical tokens); item q of a tile is the
// pair-vector g = q % vpt of token q / vpt. Element offsets within the token row:
//   e0 = h*D + fg*8 (first half of head h), e1 = e0 + D/2, with h = g / (D/16),
//   fg = g % (D/16); the table offset of the item is fg*8.
struct Item {
  int tok;   // 0..15 within the tile
  int e0;    // element offset of the first-half vector
  int f0;    // first frequency
};

__device__ __forceinline__ Item item_of(const Geom& g, int q) {
  Item it;
  it.tok = q / g.vpt;
  const int gv = q - it.tok * g.vpt;
  const int per_head = g.D >> 4;
  const int h = gv / per_head;
  it.f0 = (gv - h * per_head) * 8;
  it.e0 = h * g.D + it.f0;
  return it;
}

// ---- Work units of the tile kernels: (layer, 16-token tile, K or V, part). A part covers at
// most kPartItems pair-vectors of the tile (two per thread at 256 threads), so E up to
// 2048 never needs more than two items per thread.
constexpr int kPartItems = 512;

struct Unit {
  int li;     // layer index within the launch
  int b;      // tile (tokens b*16 .. b*16+15)
  int kv;     // 0 = K, 1 = V
  int q0;     // first item of the part
};

__host__ __device__ __forceinline__ int parts_per_tile(const Geom& g) {
  return (kTile * g.vpt + kPartItems - 1) / kPartItems;
}

__device__ __forceinline__ Unit unit_of(const Geom& g, int64_t idx, int tiles_per_layer) {
  const int parts = parts_per_tile(g);
  Unit u;
  const int part = static_cast<int>(idx % parts);
  idx /= parts;
  u.kv = static_cast<int>(idx & 1);
  idx >>= 1;
  u.li = static_cast<int>(idx / tiles_per_layer);
  u.b = static_cast<int>(idx - static_cast<int64_t>(u.li) * tiles_per_layer);
  u.q0 = part * kPartItems;
  return u;
}

// Agents handled per shared-memory chunk by the tile kernels (row table 64 x 16 x 8 B).
// Programmatic dependent launch: a kernel launched by launch_after may be scheduled while
// the stream's previous kernel is finishing. pdl_wait() returns once that kernel has
// completed and its writes are visible; a kernel calls it before it touches memory that
// earlier work may write (every kernel here that is launched this way does so first thing,
// except where its comment says what it reads before), and every CTA calls it before it
// exits, so that a kernel's completion still implies its predecessors'. pdl_trigger() lets
// the next kernel be scheduled before this one's CTAs have exited.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... P, typename... A>
inline cudaError_t launch_after(void (*kernel)(P...), unsigned grid, int threads, size_t smem,
                                cudaStream_t st, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- per-thread asynchronous copies into shared memory (cp.async, 16 bytes a copy). A
// thread that reads back only the cells it copied itself needs no barrier, only the wait.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// The same copy with an L2 cache policy (from l2_evict_first()).
__device__ __forceinline__ void cp_async16_hint(void* smem, const void* gmem, uint64_t policy) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
               "l"(policy)
               : "memory");
}
// An L2 policy under which the lines a load brings in are the first to be evicted.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// ---- mbarriers. Every wait on an mbarrier is bounded in time: a healthy copy lands in
// microseconds; after kWaitLimitNs the caller records TD_ERR_DEVICE_TIMEOUT, waits
// (bounded again) for the copies it issued and returns.
constexpr uint64_t kWaitLimitNs = 200000000ull;   // 0.2 s

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

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase with the given parity, for at most kWaitLimitNs of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < kWaitLimitNs)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

constexpr int kAgentChunk = 64;

// Row index (in elements / E) of the token at prompt position `pos` of `agent`, layer and
// kv in the paged pool, or -1 (and the error bit) when its page is unmapped.
__device__ __forceinline__ int64_t pool_row_index(const PoolDev& p, int agent, int layer,
                                                  int kv, int pos, uint32_t* err) {
  const int lp = p.p_shift >= 0 ? (pos >> p.p_shift) : pos / p.P;
  const int slot = pos - lp * p.P;
  int32_t page = -1;
  if (lp < p.max_lp) page = __ldg(p.bt + static_cast<int64_t>(agent) * p.max_lp + lp);
  if (page < 0 || page >= p.num_pages) {
    atomicOr(err, err_bit(TD_ERR_UNMAPPED_PAGE));
    return -1;
  }
  return ((static_cast<int64_t>(layer) * 2 + kv) * p.num_pages + page) * p.P + slot;
}

// Fills s_row[x * 16 + tok] with the pool row of token t0 + tok of agent agent_of(x) for
// the x < n agents of one chunk (-1 past the shared span or when unmapped).
template <typename AgentOf>
__device__ __forceinline__ void chunk_rows(const RoundDev& rd, const PoolDev& pool, int layer,
                                           int kv, int t0, int n, AgentOf agent_of,
                                           int64_t* s_row, uint32_t* err) {
  for (int idx = threadIdx.x; idx < n * kTile; idx += blockDim.x) {
    const int x = idx / kTile;
    const int t = t0 + (idx - x * kTile);
    int64_t row = -1;
    if (t < rd.S) {
      const int a = agent_of(x);
      const int j = __ldg(rd.tok_block + t);
      const int pos = __ldg(rd.off + a * rd.M + j) + t - __ldg(rd.blk_start + j);
      row = pool_row_index(pool, a, layer, kv, pos, err);
    }
    s_row[idx] = row;
  }
}

// Row address of (agent, layer, kv, position) in the paged pool, or nullptr (and the
// error bit) when the page is unmapped or out of range.
__device__ __forceinline__ uint16_t* pool_row(const PoolDev& p, int E, int agent, int layer,
                                              int kv, int pos, uint32_t* err) {
  const int lp = p.p_shift >= 0 ? (pos >> p.p_shift) : pos / p.P;
  const int slot = pos - lp * p.P;
  int32_t page = -1;
  if (lp < p.max_lp) page = __ldg(p.bt + static_cast<int64_t>(agent) * p.max_lp + lp);
  if (page < 0 || page >= p.num_pages) {
    atomicOr(err, err_bit(TD_ERR_UNMAPPED_PAGE));
    return nullptr;
  }
  const int64_t row = ((static_cast<int64_t>(layer) * 2 + kv) * p.num_pages + page) * p.P + slot;
  return p.base + row * E;
}

}  // namespace td
