"""GPU side of the parity tests: run every stage through the C ABI and compare with the
oracle chain stage by stage (each GPU stage receives the oracle's inputs for that stage,
after the previous stage was found bit-identical)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from collective_kv_cache_gb300 import runner as R
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

SENTINEL = 0xABCD


def sentinel_i16() -> int:
    return SENTINEL - 65536


def run_and_compare(cfg, seed=None, frames=(0, 1), check_guard=True):
    """Full chain on both sides; asserts bit equality of every stage's outputs."""
    orc = oracle.get()
    ch = rk.make_inputs(cfg, seed)
    rnd = ch.rnd
    # oracle chain (sentinel-filled pools so untouched rows are visible)
    pool_o = oracle.new_pool(cfg, rnd.num_pages, fill=SENTINEL)
    assert orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool_o, rnd.num_pages, rnd.block_table) == 0
    ch.k_fresh = rk.fresh_check(ch, pool_o)
    st, ch.sel, ch.dev = orc.check_select(cfg, ch.desc, pool_o, rnd.num_pages, rnd.block_table,
                                          ch.k_fresh)
    assert st == 0
    ch.master, ch.cost = orc.pick_master(cfg.n_shared, cfg.diff_block, ch.sel)
    ch.k_fresh_sel, ch.v_fresh_sel = rk.fresh_selected(ch, pool_o, ch.sel)
    ch.store = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel, ch.k_fresh_sel,
                               ch.v_fresh_sel)
    assert ch.store["status"] == 0

    dev = torch.device("cuda")
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, pool_fill=sentinel_i16())
    kc = R.to_device_bf16(ch.kc, dev)
    vc = R.to_device_bf16(ch.vc, dev)

    # stage 1
    rr.rerotate(kc, vc)
    torch.cuda.synchronize()
    got = R.bits_of(rr.pool_t)
    if check_guard:
        assert np.array_equal(got, pool_o), _first_diff(got, pool_o, "rerotate pool")
    else:
        _compare_spans(rr, ch, got, pool_o)
    del got

    # stage 2 (oracle's fresh K at the check layer)
    kf = R.to_device_bf16(ch.k_fresh, dev)
    sel = rr.check_select(kf)
    torch.cuda.synchronize()
    assert np.array_equal(rr.dev_t.cpu().numpy().view(np.uint32), ch.dev.view(np.uint32)), \
        _first_diff(rr.dev_t.cpu().numpy(), ch.dev, "deviation")
    assert np.array_equal(sel.cpu().numpy(), ch.sel), "selection differs"

    # stage 3a
    m = rr.pick_master()
    assert m == ch.master, (m, ch.master)
    assert np.array_equal(rr.cost_t.cpu().numpy(), ch.cost)

    # stage 3b (oracle's recomputed K/V at the selected tokens)
    bound = rr.candidate_bound(m)
    rr.alloc_store(max(bound, 1))
    kfs = R.to_device_bf16(ch.k_fresh_sel, dev)
    vfs = R.to_device_bf16(ch.v_fresh_sel, dev)
    nnz = rr.diff_encode(kc, vc, kfs, vfs)
    assert nnz == ch.store["nnz"], (nnz, ch.store["nnz"])
    t = rr.store_t
    assert np.array_equal(R.bits_of(t["master_k"]), ch.store["master_k"]), "master K"
    assert np.array_equal(R.bits_of(t["master_v"]), ch.store["master_v"]), "master V"
    assert np.array_equal(t["rowptr"].cpu().numpy(), ch.store["rowptr"]), "rowptr"
    assert np.array_equal(t["block_idx"].cpu().numpy()[:nnz], ch.store["idx"]), "block idx"
    assert np.array_equal(R.bits_of(t["val_k"][:nnz]), ch.store["val_k"]), "diff K values"
    assert np.array_equal(R.bits_of(t["val_v"][:nnz]), ch.store["val_v"]), "diff V values"
    _check_slots(t["slot"].cpu().numpy(), ch.store, cfg.n_agents, cfg.n_layers, rr.nb)
    s, bits = rr.get_error()
    assert s == 0 and bits == 0, (s, bits)

    # stage 4, both frames, into fresh sentinel pools
    for frame in frames:
        pool_r = oracle.new_pool(cfg, rnd.num_pages, fill=SENTINEL)
        assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents),
                                 pool_r, rnd.num_pages, rnd.block_table, frame=frame) == 0
        rr.pool_t.view(torch.int16).fill_(sentinel_i16())
        rr.fused_restore(list(range(cfg.n_agents)), frame=frame)
        torch.cuda.synchronize()
        got = R.bits_of(rr.pool_t)
        if check_guard:
            assert np.array_equal(got, pool_r), _first_diff(got, pool_r, f"restore frame {frame}")
        else:
            _compare_spans(rr, ch, got, pool_r)
        del got, pool_r
    s, bits = rr.get_error()
    assert s == 0 and bits == 0, (s, bits)
    return ch, rr


def _check_slots(slot, store, N, L, nb):
    slot = slot.reshape(N, L, nb)
    want = np.full((N, L, nb), -1, np.int64)
    rp = store["rowptr"]
    for i in range(N):
        for l in range(L):
            for r in range(rp[i * L + l], rp[i * L + l + 1]):
                want[i, l, store["idx"][r]] = r
    assert np.array_equal(slot, want), "slot map"


def _compare_spans(rr, ch, got, want):
    """Compare only the shared-span rows (used when pools are too large for a full diff)."""
    cfg = ch.cfg
    for i in range(cfg.n_agents):
        pages = ch.rnd.block_table[i, ch.pos[i] // cfg.page_size]
        slots = ch.pos[i] % cfg.page_size
        for l in range(cfg.n_layers):
            for kv in (0, 1):
                a = got[l, kv, pages, slots]
                b = want[l, kv, pages, slots]
                assert np.array_equal(a, b), (i, l, kv)


def _first_diff(a, b, what):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.shape != b.shape:
        return f"{what}: shape {a.shape} vs {b.shape}"
    bad = np.argwhere(a.view(np.uint16 if a.dtype.itemsize == 2 else np.uint32)
                      != b.view(np.uint16 if b.dtype.itemsize == 2 else np.uint32))
    return f"{what}: {len(bad)} mismatches, first at {bad[:3].tolist()}"
