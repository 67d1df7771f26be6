"""Pins of the oracle against facts that do not come from the oracle itself.

Each pin_* function takes an oracle instance and raises AssertionError on a mismatch.
test_pins_hold runs them on the oracle; test_mutants_caught (test_oracle_mutants.py) runs
them on copies of the oracle with one plausible mistake planted, and requires that at
least one pin fails for every planted mistake.

What the pins rest on:
  * IEEE / bfloat16 rounding of known values;
  * a constructive prompt layout (Figure 1 of the TokenDance review: history, then the
    shared blocks in the agent's order) instead of the offset formula;
  * textbook values cos(1), sin(1), and the float64 RoPE rotation of the test's own
    making, within the 1-bf16-ulp bound the method's tolerance states;
  * group laws of rotations: R(a)R(b) = R(a+b), R(-a)R(a) = I;
  * exact sums of squares for the deviation, brute-force sorting for the top-k and
    exhaustive set unions for the master;
  * lossless round trip of Master + diffs (the storage is block-sparse and exact);
  * closed forms of the compression ratio, and the pages' own storage table.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

THETA = 1.0e6
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rope64(x: np.ndarray, H: int, D: int, pos: float, theta: float = THETA) -> np.ndarray:
    """Float64 RoPE of one row (neox pairing), written from the rotation's definition."""
    x = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(H, D)
    half = D // 2
    f = np.arange(half, dtype=np.float64)
    ang = pos * np.power(theta, -2.0 * f / D)
    c, s = np.cos(ang), np.sin(ang)
    y = np.empty_like(x)
    y[:, :half] = x[:, :half] * c - x[:, half:] * s
    y[:, half:] = x[:, half:] * c + x[:, :half] * s
    return y.reshape(-1)


def _pair_norm(x: np.ndarray, H: int, D: int) -> np.ndarray:
    x = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(H, D)
    half = D // 2
    n = np.sqrt(x[:, :half] ** 2 + x[:, half:] ** 2)
    return np.concatenate([n, n], axis=1).reshape(-1)


def _rand_bf16(rng, n, scale=1.0):
    return synth.f32_to_bf16_bits((rng.standard_normal(n) * scale).astype(np.float32))


# --------------------------------------------------------------------------- bf16
def pin_bf16(orc):
    cases = [(1.0, 0x3F80), (1.00390625, 0x3F80), (1.0078125, 0x3F81), (1.01171875, 0x3F82),
             (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000), (math.inf, 0x7F80),
             (-math.inf, 0xFF80), (3.4028234663852886e38, 0x7F80),
             (1.1754943508222875e-38, 0x0080)]
    for x, want in cases:
        got = orc.f32_to_bf16(x)
        assert got == want, (x, hex(got), hex(want))
    h = orc.f32_to_bf16(float("nan"))
    assert (h & 0x7F80) == 0x7F80 and (h & 0x7F) != 0
    assert orc.bf16_to_f32(0x3F80) == 1.0 and orc.bf16_to_f32(0xC020) == -2.5


# --------------------------------------------------------------------------- offsets
def pin_offsets(orc):
    rng = np.random.default_rng(7)
    for trial in range(40):
        N, M = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        bl = rng.integers(1, 40, M).astype(np.int32)
        hl = rng.integers(0, 50, N).astype(np.int32)
        perm = np.stack([rng.permutation(M) for _ in range(N)]).astype(np.int32)
        off = orc.offsets(bl, hl, perm)
        for i in range(N):
            prompt = [("hist", u) for u in range(hl[i])]
            for q in range(M):
                j = int(perm[i, q])
                prompt += [(j, u) for u in range(bl[j])]
            for j in range(M):
                assert off[i, j] == prompt.index((j, 0)), (trial, i, j)
    # identity order and empty history: the canonical starts
    bl = np.array([5, 3, 9], np.int32)
    off = orc.offsets(bl, np.zeros(2, np.int32), np.array([[0, 1, 2], [0, 1, 2]], np.int32))
    assert off.tolist() == [[0, 5, 8], [0, 5, 8]]


# --------------------------------------------------------------------------- RoPE
def pin_rope_table(orc):
    c, s = orc.rope_table(0, 128, THETA)
    assert (c == 1.0).all() and (s == 0.0).all()
    c, s = orc.rope_table(1, 128, THETA)                 # f = 0 turns by 1 rad per position
    assert c[0] == np.float32(0.5403023058681398) and s[0] == np.float32(0.8414709848078965)
    c, s = orc.rope_table(1000, 64, THETA)               # f = D/4: theta^(-1/2) = 1e-3
    assert abs(c[16] - 0.5403023058681398) < 1e-6 and abs(s[16] - 0.8414709848078965) < 1e-6
    c, s = orc.rope_table(100000, 128, THETA)            # slowest frequency, f = D/2 - 1
    ang = 100000 * THETA ** (-126 / 128)
    assert abs(c[63] - math.cos(ang)) < 1e-6 and abs(s[63] - math.sin(ang)) < 1e-6


def pin_rotation_units(orc):
    H, D, a = 2, 64, 1000
    half = D // 2
    for h in range(H):
        for f in (0, 5, 16, 31):
            ang = a * THETA ** (-2 * f / D)
            for inverse in (False, True):
                sg = -1.0 if inverse else 1.0
                x = np.zeros(H * D, np.uint16)
                x[h * D + f] = 0x3F80                                   # unit on the first half
                y = synth.bf16_bits_to_f32(orc.rotate_row(x, H, D, a, THETA, inverse))
                want = np.zeros(H * D)
                want[h * D + f] = math.cos(ang)
                want[h * D + f + half] = sg * math.sin(ang)
                assert np.abs(y - want).max() <= 2.0 ** -8, (h, f, inverse)
                x = np.zeros(H * D, np.uint16)
                x[h * D + f + half] = 0x3F80                            # unit on the second half
                y = synth.bf16_bits_to_f32(orc.rotate_row(x, H, D, a, THETA, inverse))
                want = np.zeros(H * D)
                want[h * D + f] = -sg * math.sin(ang)
                want[h * D + f + half] = math.cos(ang)
                assert np.abs(y - want).max() <= 2.0 ** -8, (h, f, inverse)


def pin_rotation_bound(orc):
    """Rotated bf16 K within 1 bf16 ulp of the exact rotation: |y - y64| <= 2^-7 |pair|."""
    rng = np.random.default_rng(11)
    for H, D in ((4, 128), (2, 64), (8, 128)):
        for trial in range(20):
            x = _rand_bf16(rng, H * D)
            a = int(rng.integers(0, 40000))
            y = synth.bf16_bits_to_f32(orc.rotate_row(x, H, D, a, THETA)).astype(np.float64)
            y64 = _rope64(x, H, D, a)
            assert (np.abs(y - y64) <= 2.0 ** -7 * _pair_norm(x, H, D)).all(), (H, D, a)
            yi = synth.bf16_bits_to_f32(orc.rotate_row(x, H, D, a, THETA, True)).astype(np.float64)
            assert (np.abs(yi - _rope64(x, H, D, -a)) <= 2.0 ** -7 * _pair_norm(x, H, D)).all()
            yf = orc.rotate_row_f64(x, H, D, a, THETA)
            assert np.abs(yf - y64).max() <= 1e-9


def pin_rotation_group(orc):
    """R(b) R(a) = R(a+b) and R(-a) R(a) = I, up to the bf16 roundings in between."""
    rng = np.random.default_rng(12)
    H, D = 4, 128
    for trial in range(30):
        x = _rand_bf16(rng, H * D)
        a, b = (int(v) for v in rng.integers(0, 20000, 2))
        tol = 2.0 ** -6 * _pair_norm(x, H, D)
        ab = synth.bf16_bits_to_f32(orc.rotate_row(orc.rotate_row(x, H, D, a, THETA), H, D, b, THETA))
        direct = synth.bf16_bits_to_f32(orc.rotate_row(x, H, D, a + b, THETA))
        assert (np.abs(ab.astype(np.float64) - direct) <= tol).all()
        back = orc.rotate_row(orc.rotate_row(x, H, D, a, THETA), H, D, a, THETA, inverse=True)
        assert (np.abs(synth.bf16_bits_to_f32(back).astype(np.float64)
                       - synth.bf16_bits_to_f32(x)) <= tol).all()


# --------------------------------------------------------------------------- stage 1
def _mini_cfg(**kw):
    base = dict(name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1,
                recompute_pct=15, perturb_mode="runs", perturb_frac=(0.10, 0.20), seed=77)
    base.update(kw)
    return synth.RoundConfig(**base)


def pin_rerotate_absolute(orc):
    """Canonical-frame K (block-local positions) rerotated lands at R(absolute position)."""
    cfg = _mini_cfg()
    rnd = synth.make_round(cfg)
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    H, D, E, S, L, P = cfg.n_kv_heads, cfg.head_dim, cfg.elems, cfg.n_shared, cfg.n_layers, cfg.page_size
    rng = np.random.default_rng(5)
    raw = _rand_bf16(rng, L * S * E).reshape(L, S, E)
    start, tb, u = rk.token_layout(rnd.block_len)
    kc = np.empty_like(raw)
    for l in range(L):
        for t in range(S):
            kc[l, t] = synth.f32_to_bf16_bits(_rope64(raw[l, t], H, D, float(u[t])).astype(np.float32))
    vc = _rand_bf16(rng, L * S * E).reshape(L, S, E)
    pool = oracle.new_pool(cfg, rnd.num_pages, fill=0xABCD)
    assert orc.rerotate(cfg, desc, kc, vc, pool, rnd.num_pages, rnd.block_table) == 0
    # the test's own placement: history, then the blocks in the agent's order
    written = np.zeros(pool.shape[:4], dtype=bool)
    for i in range(cfg.n_agents):
        p = int(rnd.hist_len[i])
        for q in range(cfg.n_blocks):
            j = int(rnd.perm[i, q])
            for uu in range(int(rnd.block_len[j])):
                t = int(start[j]) + uu
                page, slot = rnd.block_table[i, p // P], p % P
                for l in range(L):
                    got = synth.bf16_bits_to_f32(pool[l, 0, page, slot].reshape(-1)).astype(np.float64)
                    want = _rope64(raw[l, t], H, D, float(p))
                    assert (np.abs(got - want) <= 2.0 ** -6 * _pair_norm(raw[l, t], H, D)).all(), (i, j, uu, l)
                    assert (pool[l, 1, page, slot].reshape(-1) == vc[l, t]).all()
                    written[l, :, page, slot] = True
                p += 1
    assert (pool[~written] == 0xABCD).all(), "rows outside the shared spans were touched"


# --------------------------------------------------------------------------- stage 2
def pin_deviation(orc):
    one = lambda x: int(synth.f32_to_bf16_bits(np.array([x], np.float32))[0])
    for E in (128, 512, 1024):
        a = np.zeros(E, np.uint16)
        b = np.zeros(E, np.uint16)
        a[0], b[1] = one(3.0), one(4.0)                      # d = (3, -4): squared distance 25
        assert orc.token_dev(a, b) == 25.0
        for e in range(E):                                   # every element is counted
            a = np.zeros(E, np.uint16)
            a[e] = one(2.0)
            assert orc.token_dev(a, np.zeros(E, np.uint16)) == 4.0, (E, e)
    rng = np.random.default_rng(3)
    for E in (128, 512, 1024):
        for trial in range(20):
            a, b = _rand_bf16(rng, E), _rand_bf16(rng, E)
            d = synth.bf16_bits_to_f32(a).astype(np.float64) - synth.bf16_bits_to_f32(b)
            exact = float(np.sum(d * d))
            got = orc.token_dev(a, b)
            assert abs(got - exact) <= 4e-6 * exact, (E, got, exact)
            assert got == orc.token_dev(b, a)


def pin_topk(orc):
    rng = np.random.default_rng(9)
    for n in (1, 7, 96, 1000):
        for k in sorted({0, 1, n // 3, n}):
            dev = (rng.integers(0, 5, n) * 0.25).astype(np.float32)   # many exact ties
            want = sorted(sorted(range(n), key=lambda t: (-float(dev[t]), t))[:k])
            assert orc.topk(dev, k).tolist() == want, (n, k)
    with pytest.raises(FloatingPointError):
        orc.topk(np.array([1.0, np.nan, 2.0], np.float32), 1)


def pin_select_recovers_perturbed(orc):
    """Tiny round: 15% of tokens carry large noise and k = ceil(15% of S): the selection
    is exactly the perturbed set of every agent."""
    cfg = synth.tiny()
    ch = rk.make_inputs(cfg, orc=orc)
    pool = oracle.new_pool(cfg, ch.rnd.num_pages)
    assert orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool, ch.rnd.num_pages, ch.rnd.block_table) == 0
    kf = rk.fresh_check(ch, pool)
    st, sel, dev = orc.check_select(cfg, ch.desc, pool, ch.rnd.num_pages, ch.rnd.block_table, kf)
    assert st == 0 and orc.last_k == 15 == sel.shape[1]
    for i in range(cfg.n_agents):
        assert sel[i].tolist() == np.nonzero(ch.rnd.perturbed[i])[0].tolist()


def pin_k_rounding(orc):
    """k = ceil(pct * S / 100): recompute fractions that do not divide S round up."""
    cfg = synth.tiny()
    ch = rk.make_inputs(cfg, orc=orc)
    pool = oracle.new_pool(cfg, ch.rnd.num_pages)
    orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool, ch.rnd.num_pages, ch.rnd.block_table)
    kf = rk.fresh_check(ch, pool)
    for pct in (0, 1, 15, 33, 50, 100):
        orc.check_select(cfg, ch.desc, pool, ch.rnd.num_pages, ch.rnd.block_table, kf, pct=pct)
        assert orc.last_k == math.ceil(pct * 96 / 100), pct


# --------------------------------------------------------------------------- stage 3a
def pin_master(orc):
    rng = np.random.default_rng(21)
    for trial in range(60):
        N, S, B = int(rng.integers(1, 7)), int(rng.integers(1, 200)), int(rng.choice([16, 32]))
        k = int(rng.integers(0, S + 1))
        k = min(k, 12)
        sel = np.stack([np.sort(rng.choice(S, k, replace=False)) for _ in range(N)]).astype(np.int32)
        sel = sel.reshape(N, k)
        blocks = [set(int(t) // B for t in sel[i]) for i in range(N)]
        cost = [sum(len(blocks[i] | blocks[m]) for i in range(N) if i != m) for m in range(N)]
        want = min(range(N), key=lambda m: (cost[m], m))
        m, got_cost = orc.pick_master(S, B, sel)
        assert got_cost.tolist() == cost and m == want, (trial, cost, m)
    sel = np.array([[3, 40], [3, 40], [3, 40]], np.int32)    # identical agents: all tie
    m, cost = orc.pick_master(64, 16, sel)
    assert m == 0 and cost.tolist() == [4, 4, 4]


def pin_master_min_dev(orc):
    """Variant master rule: the total deviation of each agent's selected tokens."""
    rng = np.random.default_rng(31)
    for trial in range(30):
        N, S = int(rng.integers(1, 7)), int(rng.integers(1, 300))
        k = int(rng.integers(0, min(S, 80) + 1))
        sel = np.stack([np.sort(rng.choice(S, k, replace=False)) for _ in range(N)]).astype(np.int32)
        sel = sel.reshape(N, k)
        dev = (rng.random((N, S)) * 100).astype(np.float32)
        m, score = orc.pick_master_min_dev(sel, dev)
        exact = [math.fsum(float(dev[i, t]) for t in sel[i]) for i in range(N)]
        for i in range(N):
            assert abs(score[i] - exact[i]) <= 1e-12 * max(1.0, abs(exact[i])), (trial, i)
        order = sorted(range(N), key=lambda i: (exact[i], i))
        if N > 1 and exact[order[1]] - exact[order[0]] > 1e-6 * max(1.0, abs(exact[order[0]])):
            assert m == order[0], (trial, m, order[0])
    # integer deviations: exact sums, ties to the lower index
    dev = np.array([[1, 2, 3, 4], [4, 3, 2, 1], [0, 0, 9, 9]], np.float32)
    sel = np.array([[0, 1], [2, 3], [0, 1]], np.int32)
    m, score = orc.pick_master_min_dev(sel, dev)
    assert score.tolist() == [3.0, 3.0, 0.0] and m == 2
    sel = np.array([[0, 1], [2, 3], [2, 3]], np.int32)
    m, score = orc.pick_master_min_dev(sel, dev)
    assert score.tolist() == [3.0, 3.0, 18.0] and m == 0
    dev[1, 2] = np.nan
    m, _ = orc.pick_master_min_dev(sel, dev)
    assert m < 0


def pin_select_group(orc):
    """Variant important set: top-k of the deviation summed over agents (integer-valued
    deviations make every float sum exact)."""
    rng = np.random.default_rng(33)
    for trial in range(25):
        N, S = int(rng.integers(1, 6)), int(rng.integers(1, 400))
        k = int(rng.integers(0, S + 1))
        dev = rng.integers(0, 6, (N, S)).astype(np.float32)       # many ties
        row, g = orc.select_group(dev, k)
        gsum = dev.astype(np.int64).sum(axis=0)
        assert (g == gsum).all()
        want = sorted(sorted(range(S), key=lambda t: (-int(gsum[t]), t))[:k])
        assert row.tolist() == want, (trial, N, S, k)
    dev = (rng.random((1, 50)) * 7).astype(np.float32)             # one agent: plain top-k
    assert orc.select_group(dev, 9)[0].tolist() == orc.topk(dev[0], 9).tolist()


# --------------------------------------------------------------------------- stage 3b / 4
def _canonical_agent_cache(orc, ch, i, l):
    """Agent i's cache at layer l in the canonical frame, built from the definition."""
    cfg = ch.cfg
    xk = ch.kc[l].copy()
    xv = ch.vc[l].copy()
    _, tb, _ = rk.token_layout(ch.rnd.block_len)
    for r, t in enumerate(ch.sel[i]):
        xk[t] = orc.rotate_row(ch.k_fresh_sel[i, l, r], cfg.n_kv_heads, cfg.head_dim,
                               int(ch.off[i, tb[t]]), cfg.rope_theta, inverse=True)
        xv[t] = ch.v_fresh_sel[i, l, r]
    return xk, xv


def pin_roundtrip(orc):
    """restore(encode(X)) == X bitwise in the canonical frame, every agent and layer;
    in the agent frame untouched tokens come back exactly as the rerotation wrote them.
    Diff blocks of 16 tokens, and of 32 tokens with 32-token pages (diff block = page)."""
    for cfg in (_mini_cfg(), _mini_cfg(diff_block=32, page_size=32)):
        _roundtrip(orc, cfg)


def _roundtrip(orc, cfg):
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, orc=orc), orc=orc, frame=1)
    N, L, S, B = cfg.n_agents, cfg.n_layers, cfg.n_shared, cfg.diff_block
    st = ch.store
    m = ch.master
    for l in range(L):
        assert st["rowptr"][m * L + l] == st["rowptr"][m * L + l + 1], "master rows must be empty"
    masks = [set(int(t) // B for t in ch.sel[i]) for i in range(N)]
    for i in range(N):
        for l in range(L):
            r0, r1 = st["rowptr"][i * L + l], st["rowptr"][i * L + l + 1]
            row = st["idx"][r0:r1].tolist()
            assert row == sorted(row) and len(set(row)) == len(row)
            if i != m:
                assert set(row) == masks[i] | masks[m], (i, l)   # every candidate differs here
    assert st["nnz"] == L * int(ch.cost[m])
    for i in range(N):
        for l in range(L):
            xk, xv = _canonical_agent_cache(orc, ch, i, l)
            gk = rk.gather_rows(ch.pool_after_restore, ch.rnd.block_table, cfg.page_size, i, l, 0, ch.pos[i])
            gv = rk.gather_rows(ch.pool_after_restore, ch.rnd.block_table, cfg.page_size, i, l, 1, ch.pos[i])
            assert (gk == xk).all() and (gv == xv).all(), (i, l)
    # agent frame
    pool = oracle.new_pool(cfg, ch.rnd.num_pages)
    assert orc.fused_restore(cfg, ch.desc, m, st, np.arange(N), pool, ch.rnd.num_pages,
                             ch.rnd.block_table, frame=0) == 0
    for i in range(N):
        not_sel = np.setdiff1d(np.arange(S), ch.sel[i])
        for l in range(L):
            got = rk.gather_rows(pool, ch.rnd.block_table, cfg.page_size, i, l, 0, ch.pos[i])
            ref = rk.gather_rows(ch.pool_after_rerotate, ch.rnd.block_table, cfg.page_size, i, l, 0, ch.pos[i])
            assert (got[not_sel] == ref[not_sel]).all(), (i, l)
            for r, t in enumerate(ch.sel[i]):
                fresh = ch.k_fresh_sel[i, l, r]
                tol = 2.0 ** -6 * _pair_norm(fresh, cfg.n_kv_heads, cfg.head_dim)
                assert (np.abs(synth.bf16_bits_to_f32(got[t]).astype(np.float64)
                               - synth.bf16_bits_to_f32(fresh)) <= tol).all()


def pin_v_only_difference(orc):
    """A block whose K equals the Master's but whose V differs is still recorded.
    One shared block at offset 0 for every agent makes the rotation the identity."""
    cfg = _mini_cfg(n_agents=3, block_lens=(48,), hist_range=(0, 0), hist_fixed=(0, 0, 0))
    ch = rk.make_inputs(cfg, orc=orc)
    N, L, S, E = cfg.n_agents, cfg.n_layers, cfg.n_shared, cfg.elems
    sel = np.tile(np.array([[3, 20, 41]], np.int32), (N, 1))
    kf = np.stack([np.stack([ch.kc[l, sel[0]] for l in range(L)])] * N)        # K unchanged
    vf = np.stack([np.stack([ch.vc[l, sel[0]] for l in range(L)])] * N)
    vf[1] ^= 1                                                                  # agent 1: V bits differ
    st = orc.diff_encode(cfg, ch.desc, 0, ch.kc, ch.vc, sel, kf, vf)
    assert st["status"] == 0
    rows = np.diff(st["rowptr"]).reshape(N, L)
    assert rows[0].sum() == 0 and rows[2].sum() == 0
    assert (rows[1] == 3).all(), rows


def pin_identical_agents(orc):
    """Agents with the same placement, selection and recomputed values need no diffs."""
    cfg = _mini_cfg(n_agents=3, hist_range=(0, 0), hist_fixed=(7, 7, 7))
    ch = rk.make_inputs(cfg, orc=orc)
    ch.rnd.perm[:] = ch.rnd.perm[0]
    ch.off = orc.offsets(*ch.desc)
    N, L = cfg.n_agents, cfg.n_layers
    sel = np.tile(np.array([[1, 2, 30, 60, 81]], np.int32), (N, 1))
    rng = np.random.default_rng(4)
    one = _rand_bf16(rng, L * 5 * cfg.elems).reshape(L, 5, cfg.elems)
    kf = np.stack([one] * N)
    vf = np.stack([one[::-1].copy()] * N)
    st = orc.diff_encode(cfg, ch.desc, 1, ch.kc, ch.vc, sel, kf, vf)
    assert st["status"] == 0 and st["nnz"] == 0
    assert orc.round_ratio(cfg, 0) == pytest.approx(
        N * (L * 82 * 128 * 4) / (L * 82 * 128 * 4 + 8 * (N * L + 1)), rel=1e-15)


def pin_empty_selection_and_capacity(orc):
    cfg = _mini_cfg(recompute_pct=0)
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, orc=orc), orc=orc, frame=1)
    assert ch.sel.shape[1] == 0 and ch.store["nnz"] == 0 and ch.master == 0
    for i in range(cfg.n_agents):                                # every agent gets Kc back
        for l in range(cfg.n_layers):
            g = rk.gather_rows(ch.pool_after_restore, ch.rnd.block_table, cfg.page_size, i, l, 0, ch.pos[i])
            assert (g == ch.kc[l]).all()
    cfg = _mini_cfg()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, orc=orc), orc=orc, restore=False)
    nnz = ch.store["nnz"]
    st = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel, ch.k_fresh_sel,
                         ch.v_fresh_sel, capacity=nnz - 1)
    assert st["status"] == oracle.ORC_ERR_CAPACITY and st["nnz"] == nnz
    assert (st["val_k"] == 0).all() and (st["val_v"] == 0).all()


# --------------------------------------------------------------------------- compression
def pin_compression(orc):
    cfg = synth.tiny()
    dense = 2 * 96 * 128 * 2 * 2
    want = 3 * dense / (dense + 24 * (16 * 128 * 4 + 4) + 8 * (3 * 2 + 1))
    assert orc.round_ratio(cfg, 24) == pytest.approx(want, rel=1e-15)
    assert orc.mirror_ratio(cfg, 8) == pytest.approx(dense / (8 * (16 * 128 * 4 + 4)), rel=1e-15)
    with open(os.path.join(GOLDEN, "storage_compression.json")) as f:
        gold = json.load(f)
    N = gold["n_agents"]
    for row in gold["rows"]:
        c7 = synth.qwen7b() if "7B" in row["model"] else synth.qwen14b()
        c7 = c7.replace(n_agents=N)
        dense = c7.n_layers * c7.n_shared * c7.elems * 4
        per_block = c7.diff_block * c7.elems * 4 + 4
        nnz_m = round(dense / (row["mirror_ratio"] * per_block))
        assert orc.mirror_ratio(c7, nnz_m) == pytest.approx(row["mirror_ratio"], rel=5e-3)
        caches = N / orc.round_ratio(c7, (N - 1) * nnz_m)
        assert round(caches, 1) == row["round_caches"], (row, caches)


# ---------------------------------------------------------------- attention from the store
def _attention_case(orc, cfg, n_q_heads, seed=None):
    """Oracle chain (encode), the agents' private histories in the pool, seeded queries,
    and the oracle's attention read from the Master and the diffs."""
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, seed, orc=orc, map_history=True), orc=orc,
                             restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages)
    rk.fill_history(cfg, rnd, pool, seed)
    agents = list(range(cfg.n_agents))
    q = synth.decode_queries(cfg, n_q_heads, agents, 0, cfg.n_layers, seed)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    st, out, lse = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool,
                                 rnd.num_pages, rnd.block_table, q, n_q_heads, scale)
    assert st == 0, st
    return ch, pool, agents, q, scale, out, lse


def pin_attention_matches_sdpa(orc):
    """Against torch's scaled_dot_product_attention (float64) on a context assembled from
    other pinned pieces: the history rows as the pool holds them, each shared position's
    canonical row from the canonical-frame restore, turned by the float64 rotation to the
    offset of the block that holds it (Figure 1's layout)."""
    torch = pytest.importorskip("torch")
    cfg = _mini_cfg(n_kv_heads=2, hist_range=(3, 40), seed=93)
    nq = 6
    ch, pool, agents, q, scale, out, lse = _attention_case(orc, cfg, nq)
    rnd, H, D, P, L = ch.rnd, cfg.n_kv_heads, cfg.head_dim, cfg.page_size, cfg.n_layers
    pool_c = oracle.new_pool(cfg, rnd.num_pages)
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents), pool_c,
                             rnd.num_pages, rnd.block_table, frame=1) == 0
    for x, a in enumerate(agents):
        h = int(rnd.hist_len[a])
        n = h + cfg.n_shared
        starts = ch.off[a]
        for l in range(L):
            K = np.empty((n, H * D))
            V = np.empty((n, H * D))
            for p in range(n):
                page, slot = rnd.block_table[a, p // P], p % P
                if p < h:
                    K[p] = synth.bf16_bits_to_f32(pool[l, 0, page, slot].reshape(-1))
                    V[p] = synth.bf16_bits_to_f32(pool[l, 1, page, slot].reshape(-1))
                else:
                    j = int(np.nonzero((starts <= p) & (p < starts + rnd.block_len))[0][0])
                    K[p] = orc.rotate_row_f64(pool_c[l, 0, page, slot].reshape(-1), H, D,
                                              int(starts[j]), cfg.rope_theta, 0)
                    V[p] = synth.bf16_bits_to_f32(pool_c[l, 1, page, slot].reshape(-1))
            qt = torch.from_numpy(synth.bf16_bits_to_f32(q[l, x]).astype(np.float64))[None, :, None, :]
            kt = torch.from_numpy(K.reshape(n, H, D).transpose(1, 0, 2)).repeat_interleave(nq // H, 0)[None]
            vt = torch.from_numpy(V.reshape(n, H, D).transpose(1, 0, 2)).repeat_interleave(nq // H, 0)[None]
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
            assert np.allclose(out[l, x], ref[0, :, 0].numpy(), rtol=0, atol=1e-10), (a, l)
            ref_lse = torch.logsumexp(scale * (qt @ kt.transpose(-1, -2)), dim=-1)
            assert np.allclose(lse[l, x], ref_lse[0, :, 0].numpy(), rtol=0, atol=1e-10), (a, l)
    # from the pages: the agent-frame restore (history kept) read as stored
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents), pool,
                             rnd.num_pages, rnd.block_table, frame=0) == 0
    q2 = synth.decode_queries(cfg, nq, agents, 0, L, seed=7)
    st, out2, _ = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool, rnd.num_pages,
                                rnd.block_table, q2, nq, scale, from_pool=True)
    assert st == 0
    for x, a in enumerate(agents):
        n = int(rnd.hist_len[a]) + cfg.n_shared
        pos = np.arange(n)
        for l in range(L):
            K = synth.bf16_bits_to_f32(rk.gather_rows(pool, rnd.block_table, P, a, l, 0, pos)).astype(np.float64)
            V = synth.bf16_bits_to_f32(rk.gather_rows(pool, rnd.block_table, P, a, l, 1, pos)).astype(np.float64)
            qt = torch.from_numpy(synth.bf16_bits_to_f32(q2[l, x]).astype(np.float64))[None, :, None, :]
            kt = torch.from_numpy(K.reshape(n, H, D).transpose(1, 0, 2)).repeat_interleave(nq // H, 0)[None]
            vt = torch.from_numpy(V.reshape(n, H, D).transpose(1, 0, 2)).repeat_interleave(nq // H, 0)[None]
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
            assert np.allclose(out2[l, x], ref[0, :, 0].numpy(), rtol=0, atol=1e-10), (a, l)


def pin_attention_single_token(orc):
    """A context of one token at position 0 (no history, one shared token, no diffs):
    the output is that token's V and the log-sum-exp its scaled score."""
    cfg = _mini_cfg(n_agents=1, n_layers=1, block_lens=(1,), hist_range=(0, 0), recompute_pct=0,
                    check_layer=0, seed=94)
    ch, pool, agents, q, scale, out, lse = _attention_case(orc, cfg, 4)
    k = synth.bf16_bits_to_f32(ch.kc[0, 0]).astype(np.float64).reshape(2, -1)
    v = synth.bf16_bits_to_f32(ch.vc[0, 0]).astype(np.float64).reshape(2, -1)
    qf = synth.bf16_bits_to_f32(q[0, 0]).astype(np.float64)
    for g in range(4):
        assert np.array_equal(out[0, 0, g], v[g // 2])
        assert abs(lse[0, 0, g] - scale * float(qf[g] @ k[g // 2])) <= 1e-12


def pin_attention_constant_values(orc):
    """Whatever the scores, a context whose V rows all equal c_h in kv head h returns c_h
    for every query head that reads head h (query head g reads head g // (n_q / H))."""
    cfg = _mini_cfg(n_kv_heads=2, hist_range=(3, 40), seed=95)
    nq, H, D = 6, 2, cfg.head_dim
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, orc=orc, map_history=True), orc=orc,
                             restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages)
    rk.fill_history(cfg, rnd, pool)
    c = synth.f32_to_bf16_bits(np.array([[0.5] * D, [-1.25] * D], np.float32)).reshape(-1)
    st = dict(ch.store)
    st["master_v"] = np.broadcast_to(c, st["master_v"].shape).copy()
    if st["nnz"]:
        st["val_v"] = np.broadcast_to(c, st["val_v"].shape).copy()
    for i, h in enumerate(rnd.hist_len):
        pos = np.arange(int(h))
        pool[:, 1, rnd.block_table[i, pos // cfg.page_size], pos % cfg.page_size] = c.reshape(H, D)
    q = synth.decode_queries(cfg, nq, range(cfg.n_agents), 0, cfg.n_layers)
    s, out, _ = orc.attention(cfg, ch.desc, ch.master, st, list(range(cfg.n_agents)), pool,
                              rnd.num_pages, rnd.block_table, q, nq, 0.3)
    assert s == 0
    want = synth.bf16_bits_to_f32(c).astype(np.float64).reshape(H, D)
    for g in range(nq):
        assert np.allclose(out[:, :, g], want[g // (nq // H)], rtol=0, atol=1e-12), g


PINS = [pin_bf16, pin_offsets, pin_rope_table, pin_rotation_units, pin_rotation_bound,
        pin_rotation_group, pin_rerotate_absolute, pin_deviation, pin_topk,
        pin_select_recovers_perturbed, pin_k_rounding, pin_master, pin_master_min_dev,
        pin_select_group, pin_roundtrip,
        pin_v_only_difference, pin_identical_agents, pin_empty_selection_and_capacity,
        pin_compression, pin_attention_matches_sdpa, pin_attention_single_token,
        pin_attention_constant_values]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pins_hold(orc, pin):
    pin(orc)
