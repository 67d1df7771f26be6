"""Parity of the variant readings with the oracle: the Master by least total deviation,
and one important set for the whole group (then encoded and restored like any other
selection)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()


def _mini(**kw):
    base = dict(name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1,
                recompute_pct=15, seed=77)
    base.update(kw)
    return synth.RoundConfig(**base)


CASES = {"tiny": synth.tiny(), "mini": _mini(), "qwen7b_3layers": synth.qwen7b().replace(n_layers=3),
         "scale64_2layers": synth.scale64().replace(n_layers=2)}


@pytest.mark.parametrize("name", list(CASES))
def test_master_by_least_total_deviation(name):
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg = CASES[name]
    ch = rk.run_oracle_chain(rk.make_inputs(cfg), restore=False)
    m_o, score_o = oracle.get().pick_master_min_dev(ch.sel, ch.dev)
    assert m_o >= 0
    rr = R.RoundRunner(cfg, ch.rnd.block_len, ch.rnd.hist_len, ch.rnd.perm, ch.rnd.block_table,
                       ch.rnd.num_pages)
    sel = torch.from_numpy(ch.sel).cuda()
    dev = torch.from_numpy(ch.dev).cuda()
    score = torch.zeros(cfg.n_agents, dtype=torch.float64, device="cuda")
    k = sel.shape[1]
    m = td.td_pick_master_min_deviation(rr.ctx.handle, rr.round, sel.data_ptr() if k else None,
                                        k, dev.data_ptr(), score.data_ptr(),
                                        rr.master_t.data_ptr(), rr.s)
    assert m == m_o
    assert np.array_equal(score.cpu().numpy().view(np.uint64), score_o.view(np.uint64))
    s, bits = rr.get_error()
    assert s == 0 and bits == 0


@pytest.mark.parametrize("name", list(CASES))
def test_group_selection_through_the_whole_path(name):
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg = CASES[name]
    orc = oracle.get()
    ch = rk.make_inputs(cfg)
    rnd = ch.rnd
    pool_o = oracle.new_pool(cfg, rnd.num_pages)
    assert orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool_o, rnd.num_pages, rnd.block_table) == 0
    ch.k_fresh = rk.fresh_check(ch, pool_o)
    st, _, dev_o = orc.check_select(cfg, ch.desc, pool_o, rnd.num_pages, rnd.block_table,
                                    ch.k_fresh)
    k = cfg.k_select
    row, g_o = orc.select_group(dev_o, k)
    sel_o = np.tile(row[None, :], (cfg.n_agents, 1)).astype(np.int32)
    m_o, cost_o = orc.pick_master(cfg.n_shared, cfg.diff_block, sel_o)
    kfs_o, vfs_o = rk.fresh_selected(ch, pool_o, sel_o)
    store_o = orc.diff_encode(cfg, ch.desc, m_o, ch.kc, ch.vc, sel_o, kfs_o, vfs_o)
    pool_r = oracle.new_pool(cfg, rnd.num_pages, fill=0x4444)
    assert orc.fused_restore(cfg, ch.desc, m_o, store_o, np.arange(cfg.n_agents), pool_r,
                             rnd.num_pages, rnd.block_table) == 0

    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, pool_fill=0x4444)
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    rr.rerotate(kc, vc)
    sel = torch.full((cfg.n_agents, k), -1, dtype=torch.int32, device="cuda")
    g = torch.zeros(cfg.n_shared, dtype=torch.float32, device="cuda")
    got_k = td.td_check_select_group(rr.ctx.handle, rr.round, cfg.check_layer, rr.pool,
                                     R.to_device_bf16(ch.k_fresh, "cuda").data_ptr(),
                                     cfg.recompute_pct, sel.data_ptr() if k else None,
                                     rr.dev_t.data_ptr(), g.data_ptr(), rr.s)
    assert got_k == k
    torch.cuda.synchronize()
    assert np.array_equal(g.cpu().numpy().view(np.uint32), g_o.view(np.uint32))
    assert np.array_equal(sel.cpu().numpy(), sel_o)
    m = rr.pick_master(sel)
    assert m == m_o and np.array_equal(rr.cost_t.cpu().numpy(), cost_o)
    rr.alloc_store(max(rr.candidate_bound(m), 1))
    nnz = rr.diff_encode(kc, vc, R.to_device_bf16(kfs_o, "cuda"), R.to_device_bf16(vfs_o, "cuda"),
                         sel=sel)
    assert nnz == store_o["nnz"]
    assert np.array_equal(R.bits_of(rr.store_t["val_k"][:nnz]), store_o["val_k"])
    rr.pool_t.view(torch.int16).fill_(0x4444)
    rr.fused_restore(list(range(cfg.n_agents)))
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(rr.pool_t), pool_r)
    s, bits = rr.get_error()
    assert s == 0 and bits == 0
