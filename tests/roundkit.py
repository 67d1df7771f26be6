"""Test-side assembly of a synthetic round and of the oracle's full chain.

The synthetic 'recomputed' K/V are the reused values plus the generator's noise, which is
how the workloads describe them (fresh K = reused K + small noise, large noise on the
perturbed tokens). Everything here runs on the CPU through the oracle.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

import oracle as _oracle
from collective_kv_cache_gb300 import synth


token_layout = synth.token_layout
positions = synth.positions
gather_rows = synth.gather_rows


@dataclasses.dataclass
class Chain:
    cfg: synth.RoundConfig
    rnd: synth.Round
    desc: tuple                 # (block_len, hist_len, perm)
    off: np.ndarray
    pos: np.ndarray             # [N][S]
    kc: np.ndarray
    vc: np.ndarray
    pool_after_rerotate: Optional[np.ndarray] = None
    k_fresh: Optional[np.ndarray] = None      # [N][S][E]
    sel: Optional[np.ndarray] = None
    dev: Optional[np.ndarray] = None
    master: Optional[int] = None
    cost: Optional[np.ndarray] = None
    k_fresh_sel: Optional[np.ndarray] = None  # [N][L][k][E]
    v_fresh_sel: Optional[np.ndarray] = None
    store: Optional[dict] = None
    pool_after_restore: Optional[np.ndarray] = None


def make_inputs(cfg: synth.RoundConfig, seed: Optional[int] = None, orc=None,
                map_history: bool = False) -> Chain:
    orc = orc or _oracle.get()
    rnd = synth.make_round(cfg, seed, map_history=map_history)
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    off = orc.offsets(*desc)
    kc, vc = synth.canonical_kv(cfg, seed)
    return Chain(cfg, rnd, desc, off, positions(off, rnd.block_len), kc, vc)


def fill_history(cfg: synth.RoundConfig, rnd: synth.Round, pool: np.ndarray,
                 seed: Optional[int] = None) -> None:
    """Writes every agent's private-history K/V (synth.history_rows) into its pages."""
    P = cfg.page_size
    for i, h in enumerate(rnd.hist_len):
        h = int(h)
        if h == 0:
            continue
        pos = np.arange(h)
        pages = rnd.block_table[i, pos // P]
        assert (pages >= 0).all()
        for l in range(cfg.n_layers):
            for kv, name in ((0, "K"), (1, "V")):
                rows = synth.history_rows(cfg, i, l, name, h, seed)
                pool[l, kv, pages, pos % P] = rows.reshape(h, cfg.n_kv_heads, cfg.head_dim)


def fresh_check(ch: Chain, pool: np.ndarray) -> np.ndarray:
    """Synthetic recomputed K at the check layer: reused K + check-layer noise."""
    return synth.recompute_check(ch.cfg, ch.rnd, ch.pos, pool)


def fresh_selected(ch: Chain, pool: np.ndarray, sel: np.ndarray):
    """Synthetic recomputed K (agent frame) and V at the selected tokens of every layer."""
    return synth.recompute_selected(ch.cfg, ch.rnd, ch.pos, pool, ch.vc, sel)


def run_oracle_chain(ch: Chain, restore: bool = True, orc=None, frame: int = 0) -> Chain:
    orc = orc or _oracle.get()
    cfg, rnd = ch.cfg, ch.rnd
    pool = _oracle.new_pool(cfg, rnd.num_pages)
    st = orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool, rnd.num_pages, rnd.block_table)
    assert st == 0, st
    ch.pool_after_rerotate = pool.copy()
    ch.k_fresh = fresh_check(ch, pool)
    st, ch.sel, ch.dev = orc.check_select(cfg, ch.desc, pool, rnd.num_pages, rnd.block_table,
                                          ch.k_fresh)
    assert st == 0, st
    ch.master, ch.cost = orc.pick_master(cfg.n_shared, cfg.diff_block, ch.sel)
    ch.k_fresh_sel, ch.v_fresh_sel = fresh_selected(ch, pool, ch.sel)
    ch.store = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel, ch.k_fresh_sel,
                               ch.v_fresh_sel)
    assert ch.store["status"] == 0, ch.store["status"]
    if restore:
        pool2 = _oracle.new_pool(cfg, rnd.num_pages)
        st = orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents),
                               pool2, rnd.num_pages, rnd.block_table, frame=frame)
        assert st == 0, st
        ch.pool_after_restore = pool2
    return ch
