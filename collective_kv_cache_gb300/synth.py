"""Seeded synthetic All-Gather rounds: the inputs both the CUDA path and the oracle consume.

This module draws random numbers and integer placements only. It holds none of the
method's arithmetic (no rotation, no deviation, no selection, no diffing): a caller that
needs a "freshly recomputed" K builds it from the reused K it already has plus the noise
drawn here.

Workload shape (TokenDance, "Summary — Motivation" and Figure 1): agent i's prompt is its
private history H_i followed by the N shared output blocks in an agent-specific order
Pi_i. The pages measure on GenerativeAgents / AgentSociety traces with Qwen2.5-7B/14B;
those traces and weights are not available, so the rounds below stand in for them with
the model shapes (layers, KV heads, head_dim), the block and history lengths and the
perturbation fractions of the five workloads this library is tested on.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used counter-style: element n of a stream with key K is
mix(K + (n+1)*GAMMA). Normals are an Irwin-Hall sum of four 16-bit uniforms, scaled to
unit variance in float64 (exact integer sum, one IEEE division), so every machine draws
identical bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

_U = np.uint64
GAMMA = _U(0x9E3779B97F4A7C15)
_M1 = _U(0xBF58476D1CE4E5B9)
_M2 = _U(0x94D049BB133111EB)
# Irwin-Hall(4) of uniform integers on [0, 65535]: mean 2*65535, variance 4*(65536^2-1)/12
_IH_MEAN = 2 * 65535
_IH_SD = math.sqrt(4.0 * (65536.0 * 65536.0 - 1.0) / 12.0)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> _U(30))) * _M1
    z = (z ^ (z >> _U(27))) * _M2
    return z ^ (z >> _U(31))


def _tag(s) -> int:
    if isinstance(s, str):
        h = 1469598103934665603  # multiplicative byte hash of the tag (FNV's prime)
        for ch in s.encode():
            h = ((h ^ ch) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
        return h
    return int(s) & 0xFFFFFFFFFFFFFFFF


def stream_key(seed: int, *ids) -> np.uint64:
    """Key of the sub-stream named by (seed, ids...)."""
    k = _mix(np.array([_tag(seed)], dtype=_U) + GAMMA)
    for x in ids:
        k = _mix(k ^ _mix(np.array([_tag(x)], dtype=_U) + GAMMA))
    return k[0]


def uniform_u64(key, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 output for each counter (any integer array, >= 0)."""
    c = np.asarray(counters, dtype=_U)
    return _mix(_U(key) + (c + _U(1)) * GAMMA)


def normal_f64(key, counters: np.ndarray) -> np.ndarray:
    """Approximately N(0, 1) per counter: Irwin-Hall(4) of 16-bit uniforms, unit variance."""
    u = uniform_u64(key, counters)
    m = _U(0xFFFF)
    s = (u & m) + ((u >> _U(16)) & m) + ((u >> _U(32)) & m) + (u >> _U(48))
    return (s.astype(np.int64) - _IH_MEAN).astype(np.float64) / _IH_SD


# ---------------------------------------------------------------- the same draws in torch
# SplitMix64 on int64 tensors: products wrap modulo 2^64 like uint64, right shifts are made
# logical by masking, so CPU and GPU tensors give the bits numpy gives.
_T_GAMMA = int(np.array(GAMMA).astype(np.int64))
_T_M1 = int(np.array(_M1).astype(np.int64))
_T_M2 = int(np.array(_M2).astype(np.int64))


def _t_shr(x, s: int):
    return (x >> s) & ((1 << (64 - s)) - 1)


def _t_mix(z):
    z = (z ^ _t_shr(z, 30)) * _T_M1
    z = (z ^ _t_shr(z, 27)) * _T_M2
    return z ^ _t_shr(z, 31)


def normal_torch64(key, counters, scale: float = 1.0):
    """normal_f64(key, counters) * scale in float64, computed by torch on the counters'
    device (counters: an int64 tensor)."""
    import torch
    k = int(np.array(key, dtype=np.uint64).astype(np.int64))
    u = _t_mix(k + (counters + 1) * _T_GAMMA)
    m = 0xFFFF
    s = (u & m) + (_t_shr(u, 16) & m) + (_t_shr(u, 32) & m) + _t_shr(u, 48)
    return (s - _IH_MEAN).to(torch.float64) / _IH_SD * scale


def normal_torch(key, counters, scale: float = 1.0):
    """normal_torch64 rounded to float32."""
    import torch
    return normal_torch64(key, counters, scale).to(torch.float32)


def canonical_torch(cfg: "RoundConfig", kv: str, layer: int, device, seed=None):
    """One layer of canonical K or V, [S][E] bf16, on `device` (same bits as canonical_kv)."""
    import torch
    seed = cfg.seed if seed is None else seed
    S, E = cfg.n_shared, cfg.elems
    ctr = torch.arange(S * E, dtype=torch.int64, device=device)
    x = normal_torch(stream_key(seed, "canon", kv, layer), ctr)
    return x.to(torch.bfloat16).reshape(S, E)


def noise_rows_torch(seed, tag, agent, layer, tokens, perturbed_rows, E):
    """_noise_rows on torch tensors (tokens, perturbed_rows on the target device)."""
    import torch
    lane = torch.arange(E, dtype=torch.int64, device=tokens.device)
    ctr = (tokens.to(torch.int64)[:, None] * E + lane[None, :]).reshape(-1)
    out = normal_torch64(stream_key(seed, tag, "small", agent, layer), ctr,
                         1.0e-3).reshape(len(tokens), E)
    if bool(perturbed_rows.any()):
        tp = tokens.to(torch.int64)[perturbed_rows]
        ctr_big = (tp[:, None] * E + lane[None, :]).reshape(-1)
        big = normal_torch64(stream_key(seed, tag, "big", agent, layer), ctr_big,
                             0.5).reshape(-1, E)
        out[perturbed_rows] += big
    return out.to(torch.float32)


def history_rows(cfg: "RoundConfig", agent: int, layer: int, kv: str, n: int,
                 seed=None) -> np.ndarray:
    """K or V of an agent's first n private-history positions at one layer, [n][E] bf16
    bits, N(0, 1) (as stored in the pool: K already in the agent frame)."""
    seed = cfg.seed if seed is None else seed
    ctr = np.arange(n * cfg.elems, dtype=np.int64)
    x = normal_f64(stream_key(seed, "hist", kv, agent, layer), ctr).astype(np.float32)
    return f32_to_bf16_bits(x).reshape(n, cfg.elems)


def history_torch(cfg: "RoundConfig", agent: int, layer: int, kv: str, n: int, device,
                  seed=None):
    """history_rows on `device`, [n][E] bf16 (same bits)."""
    import torch
    seed = cfg.seed if seed is None else seed
    ctr = torch.arange(n * cfg.elems, dtype=torch.int64, device=device)
    x = normal_torch(stream_key(seed, "hist", kv, agent, layer), ctr)
    return x.to(torch.bfloat16).reshape(n, cfg.elems)


def decode_queries(cfg: "RoundConfig", n_q_heads: int, agents, layer_begin: int, layer_end: int,
                   seed=None) -> np.ndarray:
    """One decode query per (layer, agent, query head), agent frame, N(0, 1):
    [nl][len(agents)][n_q_heads][D] bf16 bits."""
    seed = cfg.seed if seed is None else seed
    D = cfg.head_dim
    out = np.empty((layer_end - layer_begin, len(agents), n_q_heads, D), dtype=np.uint16)
    ctr = np.arange(n_q_heads * D, dtype=np.int64)
    for li in range(layer_end - layer_begin):
        for x, a in enumerate(agents):
            q = normal_f64(stream_key(seed, "query", int(a), layer_begin + li), ctr)
            out[li, x] = f32_to_bf16_bits(q.astype(np.float32)).reshape(n_q_heads, D)
    return out


def round_prompts(rnd: "Round", sep: int, vocab: int = 150000, seed=None):
    """Token prompts of a round: agent i's history (hist_len[i] tokens), then the shared
    blocks in its order, each block starting with the separator `sep` followed by its
    block_len - 1 content tokens (the same for every agent). Tokens in [1, vocab), never
    `sep`. Returns a list of int32 arrays."""
    cfg = rnd.cfg
    seed = cfg.seed if seed is None else seed

    def toks(key, n):
        t = randint(key, np.arange(n), 1, vocab - 2).astype(np.int32)
        return np.where(t >= sep, t + 1, t).astype(np.int32)

    blocks = []
    for j, L in enumerate(rnd.block_len):
        body = toks(stream_key(seed, "block-tokens", j), int(L) - 1)
        blocks.append(np.concatenate([np.array([sep], np.int32), body]))
    out = []
    for i, h in enumerate(rnd.hist_len):
        parts = [toks(stream_key(seed, "hist-tokens", i), int(h))]
        parts += [blocks[j] for j in rnd.perm[i]]
        out.append(np.concatenate(parts).astype(np.int32))
    return out


def randint(key, counters, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive)."""
    span = _U(hi - lo + 1)
    return (uniform_u64(key, counters) % span).astype(np.int64) + lo


# ---------------------------------------------------------------- bf16 storage helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even; NaN stays NaN."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    is_nan = (b & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    r = (b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    r = np.where(is_nan, (b >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- workload descriptions
@dataclasses.dataclass(frozen=True)
class RoundConfig:
    """One synthetic All-Gather round: model shape, placement and perturbation recipe."""

    name: str
    n_agents: int
    n_layers: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    block_lens: tuple                 # length of each shared output block, canonical order
    hist_range: tuple                 # (lo, hi) inclusive, uniform; ignored if hist_fixed
    hist_fixed: Optional[tuple] = None
    check_layer: int = 1
    recompute_pct: int = 15
    perturb_mode: str = "runs"        # "runs": clustered runs of 1..64 tokens; "uniform"
    perturb_frac: tuple = (0.10, 0.20)  # per-agent fraction, uniform on [lo, hi]
    rope_theta: float = 1.0e6
    diff_block: int = 16
    pool_bytes: Optional[int] = None  # paged pool size; None = exactly the pages needed
    seed: int = 1000
    n_q_heads: int = 0                # decode query heads (0: as many as kv heads)

    @property
    def n_blocks(self) -> int:
        return len(self.block_lens)

    @property
    def n_shared(self) -> int:
        return int(sum(self.block_lens))

    @property
    def elems(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def k_select(self) -> int:
        return (self.recompute_pct * self.n_shared + 99) // 100

    def replace(self, **kw) -> "RoundConfig":
        return dataclasses.replace(self, **kw)


def tiny() -> RoundConfig:
    return RoundConfig(
        name="tiny_n3_l2_h2x64_s96", n_agents=3, n_layers=2, n_kv_heads=2, head_dim=64,
        page_size=16, block_lens=(32, 32, 32), hist_range=(0, 0), hist_fixed=(5, 17, 40),
        check_layer=0, recompute_pct=15, perturb_mode="uniform", perturb_frac=(0.15, 0.15),
        seed=1000)


def qwen7b() -> RoundConfig:
    return RoundConfig(
        name="qwen2.5-7b_n10_l28_h4x128_s2560", n_agents=10, n_layers=28, n_kv_heads=4,
        head_dim=128, page_size=16, block_lens=(256,) * 10, hist_range=(500, 4000),
        check_layer=1, recompute_pct=15, seed=1001, n_q_heads=28)


def qwen14b() -> RoundConfig:
    return RoundConfig(
        name="qwen2.5-14b_n10_l48_h8x128_s5120", n_agents=10, n_layers=48, n_kv_heads=8,
        head_dim=128, page_size=16, block_lens=(512,) * 10, hist_range=(1000, 8000),
        check_layer=1, recompute_pct=15, seed=1002, n_q_heads=40)


def scale64() -> RoundConfig:
    return RoundConfig(
        name="qwen2.5-7b_n64_l28_h4x128_s8192", n_agents=64, n_layers=28, n_kv_heads=4,
        head_dim=128, page_size=16, block_lens=(128,) * 64, hist_range=(0, 16384),
        check_layer=1, recompute_pct=15, seed=1003, n_q_heads=28)


def density(pct: int, page_size: int = 16, pool_bytes: Optional[int] = 120 * 10**9) -> RoundConfig:
    f = pct / 100.0
    return RoundConfig(
        name=f"qwen2.5-14b_n32_l48_h8x128_s16384_p{pct}_pg{page_size}", n_agents=32,
        n_layers=48, n_kv_heads=8, head_dim=128, page_size=page_size,
        block_lens=(512,) * 32, hist_range=(1000, 8000), check_layer=1, recompute_pct=pct,
        perturb_frac=(f, f), pool_bytes=pool_bytes, seed=1004, n_q_heads=40)


CONFIGS = {"tiny": tiny, "qwen7b": qwen7b, "qwen14b": qwen14b, "scale64": scale64}


# ---------------------------------------------------------------- the round itself
@dataclasses.dataclass
class Round:
    cfg: RoundConfig
    block_len: np.ndarray      # [M] int32
    hist_len: np.ndarray       # [N] int32
    perm: np.ndarray           # [N, M] int32: perm[i, q] = block at slot q of agent i
    perturbed: np.ndarray      # [N, S] bool: tokens whose fresh K/V carry large noise
    block_table: np.ndarray    # [N, max_lp] int32, -1 = unmapped
    num_pages: int


def _perturbed_mask(cfg: RoundConfig, seed: int) -> np.ndarray:
    N, S = cfg.n_agents, cfg.n_shared
    out = np.zeros((N, S), dtype=bool)
    lo, hi = cfg.perturb_frac
    for i in range(N):
        cnt_lo = int(math.ceil(lo * S - 1e-9))
        cnt_hi = int(math.floor(hi * S + 1e-9))
        cnt_hi = max(cnt_hi, cnt_lo)
        target = int(randint(stream_key(seed, "pert-count", i), [0], cnt_lo, cnt_hi)[0])
        target = min(target, S)
        if cfg.perturb_mode == "uniform":
            keys = uniform_u64(stream_key(seed, "pert-uniform", i), np.arange(S))
            out[i, np.argsort(keys, kind="stable")[:target]] = True
            continue
        key = stream_key(seed, "pert-runs", i)
        marked, n = 0, 0
        while marked < target:
            r = uniform_u64(key, [n])[0]
            n += 1
            run = int(r % _U(64)) + 1
            start = int((r >> _U(8)) % _U(max(S - run + 1, 1)))
            for t in range(start, min(start + run, S)):
                if not out[i, t]:
                    out[i, t] = True
                    marked += 1
                    if marked == target:
                        break
    return out


def make_round(cfg: RoundConfig, seed: Optional[int] = None,
               map_history: bool = False) -> Round:
    """Round descriptor, perturbation mask and a randomly permuted page table.

    Pages that hold only private history stay unmapped (-1) unless map_history.
    """
    seed = cfg.seed if seed is None else seed
    N, M, S, P = cfg.n_agents, cfg.n_blocks, cfg.n_shared, cfg.page_size
    block_len = np.asarray(cfg.block_lens, dtype=np.int32)
    if cfg.hist_fixed is not None:
        hist = np.asarray(cfg.hist_fixed, dtype=np.int32)
    else:
        hist = randint(stream_key(seed, "hist"), np.arange(N), *cfg.hist_range).astype(np.int32)
    perm = np.empty((N, M), dtype=np.int32)
    for i in range(N):
        keys = uniform_u64(stream_key(seed, "perm", i), np.arange(M))
        perm[i] = np.argsort(keys, kind="stable")
    perturbed = _perturbed_mask(cfg, seed)

    max_lp = int(max((int(h) + S + P - 1) // P for h in hist))
    first = [0 if map_history else int(h) // P for h in hist]
    last = [(int(h) + S - 1) // P for h in hist]
    need = sum(l - f + 1 for f, l in zip(first, last))
    page_bytes = cfg.n_layers * 2 * P * cfg.elems * 2
    num_pages = need if cfg.pool_bytes is None else max(need, cfg.pool_bytes // page_bytes)
    phys = np.argsort(uniform_u64(stream_key(seed, "pages"), np.arange(num_pages)),
                      kind="stable").astype(np.int32)
    bt = np.full((N, max_lp), -1, dtype=np.int32)
    c = 0
    for i in range(N):
        n_i = last[i] - first[i] + 1
        bt[i, first[i]:last[i] + 1] = phys[c:c + n_i]
        c += n_i
    return Round(cfg, block_len, hist, perm, perturbed, bt, int(num_pages))


# ---------------------------------------------------------------- tensors
def canonical_kv(cfg: RoundConfig, seed: Optional[int] = None, layers=None,
                 chunk_rows: int = 4096):
    """Canonical-frame K and V, [L][S][E] bf16 bits (uint16), entries ~ N(0, 1)."""
    seed = cfg.seed if seed is None else seed
    L, S, E = cfg.n_layers, cfg.n_shared, cfg.elems
    layers = range(L) if layers is None else layers
    out = []
    for kv in ("K", "V"):
        arr = np.empty((len(layers), S, E), dtype=np.uint16)
        for li, l in enumerate(layers):
            key = stream_key(seed, "canon", kv, l)
            for t0 in range(0, S, chunk_rows):
                t1 = min(S, t0 + chunk_rows)
                ctr = np.arange(t0 * E, t1 * E, dtype=np.uint64)
                arr[li, t0:t1] = f32_to_bf16_bits(
                    normal_f64(key, ctr).astype(np.float32)).reshape(t1 - t0, E)
        out.append(arr)
    return out[0], out[1]


def _noise_rows(seed, tag, agent, layer, tokens, perturbed_rows, E):
    """Noise for whole token rows: N(0, 1e-3) everywhere plus N(0, 0.5) on perturbed rows."""
    tokens = np.asarray(tokens, dtype=np.int64)
    pr = np.asarray(perturbed_rows, dtype=bool)
    lane = np.arange(E, dtype=np.int64)[None, :]
    ctr = (tokens[:, None] * E + lane).reshape(-1)
    out = (normal_f64(stream_key(seed, tag, "small", agent, layer), ctr) * 1.0e-3).reshape(len(tokens), E)
    if pr.any():
        ctr_big = (tokens[pr][:, None] * E + lane).reshape(-1)
        out[pr] += (normal_f64(stream_key(seed, tag, "big", agent, layer), ctr_big) * 0.5).reshape(-1, E)
    return out.astype(np.float32)


def check_noise(rnd: Round, seed: Optional[int] = None) -> np.ndarray:
    """[N][S][E] float32: added to each agent's reused K at the check layer to make the
    'fresh' K the selection compares against."""
    cfg = rnd.cfg
    seed = cfg.seed if seed is None else seed
    N, S, E = cfg.n_agents, cfg.n_shared, cfg.elems
    out = np.empty((N, S, E), dtype=np.float32)
    for i in range(N):
        out[i] = _noise_rows(seed, "chk", i, cfg.check_layer, np.arange(S), rnd.perturbed[i], E)
    return out


def selected_noise(rnd: Round, sel: np.ndarray, layers=None, seed: Optional[int] = None):
    """Noise for the fresh K and V at the selected tokens of every layer:
    two float32 arrays [N][len(layers)][k][E], keyed by (agent, layer, token), so the
    values do not depend on how the selection is stored."""
    cfg = rnd.cfg
    seed = cfg.seed if seed is None else seed
    layers = range(cfg.n_layers) if layers is None else layers
    N, E = cfg.n_agents, cfg.elems
    k = sel.shape[1]
    nk = np.empty((N, len(layers), k, E), dtype=np.float32)
    nv = np.empty_like(nk)
    for i in range(N):
        pr = rnd.perturbed[i, sel[i]] if k else np.zeros(0, bool)
        for li, l in enumerate(layers):
            nk[i, li] = _noise_rows(seed, "selK", i, l, sel[i], pr, E)
            nv[i, li] = _noise_rows(seed, "selV", i, l, sel[i], pr, E)
    return nk, nv


def add_noise_bf16(base_bits: np.ndarray, noise: np.ndarray) -> np.ndarray:
    """bf16(float32(base) + noise), round to nearest even: a synthetic 'recomputed' value."""
    return f32_to_bf16_bits(bf16_bits_to_f32(base_bits) + noise)


# ---------------------------------------------------------------- synthetic recompute on the host
# The recomputed K/V the workloads describe (reused value + the generator's noise), built
# from a host copy of a pool. Only array layout and the noise model: positions come from
# the caller's block offsets.
def token_layout(block_len):
    """Canonical start of each block, and the block and local index of each token."""
    bl = np.asarray(block_len, dtype=np.int64)
    start = np.concatenate([[0], np.cumsum(bl)[:-1]])
    tok_block = np.repeat(np.arange(len(bl)), bl)
    u = np.arange(int(bl.sum())) - start[tok_block]
    return start, tok_block, u


def positions(off: np.ndarray, block_len) -> np.ndarray:
    """[N][S]: prompt position of canonical token t in agent i, from block offsets off[N][M]."""
    _, tb, u = token_layout(block_len)
    return off[:, tb] + u[None, :]


def gather_rows(pool: np.ndarray, block_table: np.ndarray, P: int, agent: int, layer: int,
                kv: int, pos: np.ndarray) -> np.ndarray:
    """Rows of one agent's paged cache (host array [L][2][pages][P][H][D]) at prompt
    positions pos -> [len(pos)][E]."""
    pages = block_table[agent, pos // P]
    assert (pages >= 0).all()
    rows = pool[layer, kv, pages, pos % P]
    return rows.reshape(len(pos), pool.shape[4] * pool.shape[5])


def recompute_check(cfg: RoundConfig, rnd: Round, pos: np.ndarray, pool: np.ndarray) -> np.ndarray:
    """Recomputed K at the check layer, [N][S][E] bf16 bits: reused K + check-layer noise."""
    noise = check_noise(rnd)
    out = np.empty((cfg.n_agents, cfg.n_shared, cfg.elems), dtype=np.uint16)
    for i in range(cfg.n_agents):
        reused = gather_rows(pool, rnd.block_table, cfg.page_size, i, cfg.check_layer, 0, pos[i])
        out[i] = add_noise_bf16(reused, noise[i])
    return out


def recompute_selected(cfg: RoundConfig, rnd: Round, pos: np.ndarray, pool: np.ndarray,
                       vc: np.ndarray, sel: np.ndarray):
    """Recomputed K (agent frame, from the pool) and V (from the canonical V) at the
    selected tokens of every layer: [N][L][k][E] bf16 bits each."""
    nk, nv = selected_noise(rnd, sel)
    N, L, k, E = cfg.n_agents, cfg.n_layers, sel.shape[1], cfg.elems
    kf = np.empty((N, L, k, E), dtype=np.uint16)
    vf = np.empty((N, L, k, E), dtype=np.uint16)
    for i in range(N):
        for l in range(L):
            reused = gather_rows(pool, rnd.block_table, cfg.page_size, i, l, 0, pos[i, sel[i]])
            kf[i, l] = add_noise_bf16(reused, nk[i, l])
            vf[i, l] = add_noise_bf16(vc[l, sel[i]], nv[i, l])
    return kf, vf
