"""td_check_select_noalloc: the selection entry point for callers that may not allocate
device memory (code under an allocator that forbids cudaMalloc, or a process whose device
footprint must stay fixed after start-up). On consecutive calls that reuse its fixed
scratch it must give exactly the oracle's selection and exactly what td_check_select gives
on the same inputs, and it must refuse rounds that do not fit its scratch.

Collected last on purpose, so that a run that stops at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()
    from collective_kv_cache_gb300 import td
    return td


def _oracle_round(cfg):
    """The oracle's re-rotated pool, recomputed K at the check layer and selection, with the
    same pool and K on the device."""
    from collective_kv_cache_gb300 import runner as R
    orc = oracle.get()
    ch = rk.make_inputs(cfg)
    rnd = ch.rnd
    pool_o = oracle.new_pool(cfg, rnd.num_pages)
    assert orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool_o, rnd.num_pages, rnd.block_table) == 0
    k_fresh = rk.fresh_check(ch, pool_o)
    st, sel, _ = orc.check_select(cfg, ch.desc, pool_o, rnd.num_pages, rnd.block_table, k_fresh)
    assert st == 0
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages)
    rr.pool_t.copy_(R.to_device_bf16(pool_o, "cuda").view(rr.pool_t.shape))
    kf = R.to_device_bf16(k_fresh, "cuda")
    return rr, kf, sel


def _mini(**kw):
    base = dict(name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1,
                recompute_pct=15, seed=77)
    base.update(kw)
    return synth.RoundConfig(**base)


def test_noalloc_matches_oracle_and_context_path_on_consecutive_calls(lib):
    td = lib
    rounds = [_oracle_round(_mini()),
              _oracle_round(synth.qwen7b().replace(n_layers=3)),
              _oracle_round(_mini(diff_block=32, page_size=32, seed=78))]
    # A, B, C, A: later calls find the previous call's contents in the scratch
    for idx in (0, 1, 2, 0):
        rr, kf, sel_orc = rounds[idx]
        cfg = rr.cfg
        sel = torch.full(sel_orc.shape, -7, dtype=torch.int32, device="cuda")
        s, k, bits = td.td_check_select_noalloc(td.make_shape(cfg), rr.round, cfg.check_layer,
                                                rr.pool, kf.data_ptr(), cfg.recompute_pct,
                                                sel.data_ptr(), rr.s)
        assert s == td.TD_OK and bits == 0, (s, bits)
        assert k == sel_orc.shape[1]
        torch.cuda.synchronize()
        assert np.array_equal(sel.cpu().numpy(), sel_orc), f"round {idx}: differs from the oracle"
        sel_ctx = rr.check_select(kf)
        torch.cuda.synchronize()
        assert torch.equal(sel, sel_ctx), f"round {idx}: differs from td_check_select"


def test_noalloc_rejects_rounds_beyond_its_scratch(lib):
    td = lib
    cfg = synth.RoundConfig(name="big", n_agents=64, n_layers=2, n_kv_heads=1, head_dim=16,
                            page_size=16, block_lens=(20000,), hist_range=(0, 0),
                            hist_fixed=(0,) * 64, check_layer=0)
    rnd = td.make_round(np.array([20000]), np.zeros(64, np.int32), np.zeros((64, 1), np.int32))
    pool_t = torch.zeros((2, 2, 4, 16, 1, 16), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    kf = torch.zeros((16,), dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    s, _, _ = td.td_check_select_noalloc(td.make_shape(cfg), rnd, 0, td.make_paged(pool_t, bt),
                                         kf.data_ptr(), 15, sel.data_ptr())
    assert s == td.TD_ERR_SCRATCH_LIMIT
