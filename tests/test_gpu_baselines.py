"""The in-run comparison baselines compute what the path computes.

Serial per-request PIC (one re-rotation and one check-layer selection per agent, each
re-reading the canonical K/V) must leave the same pages, deviations and selections as the
collective launch; the dense restore (materialise each agent's cache, then re-rotate it
into its pages) must leave the same pages as the fused restore, and its materialised cache
must equal the oracle's canonical-frame restore at the agent's positions.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

pytestmark = pytest.mark.gpu

SENTINEL_I16 = 0x4444


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()


def _mini(**kw):
    base = dict(name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=24,
                block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1,
                recompute_pct=15, seed=91)
    base.update(kw)
    return synth.RoundConfig(**base)


CASES = {"tiny": synth.tiny(), "mini": _mini(), "mini_b32": _mini(diff_block=32, page_size=32),
         "qwen7b_3layers": synth.qwen7b().replace(n_layers=3)}


def _runner(cfg, rnd):
    from collective_kv_cache_gb300 import runner as R
    return R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                         rnd.num_pages, pool_fill=SENTINEL_I16)


@pytest.mark.parametrize("name", list(CASES))
def test_serial_pic_equals_collective(name):
    from collective_kv_cache_gb300 import runner as R
    cfg = CASES[name]
    ch = rk.run_oracle_chain(rk.make_inputs(cfg), restore=False)
    rnd = ch.rnd
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    kf = R.to_device_bf16(ch.k_fresh, "cuda")
    a, b = _runner(cfg, rnd), _runner(cfg, rnd)
    a.rerotate(kc, vc)
    sel_a = a.check_select(kf)
    b.serial_pic(kc, vc, kf)
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(a.pool_t), R.bits_of(b.pool_t))
    assert np.array_equal(sel_a.cpu().numpy(), b.sel_t.cpu().numpy())
    assert np.array_equal(b.sel_t.cpu().numpy(), ch.sel)
    assert np.array_equal(b.dev_t.cpu().numpy().view(np.uint32), ch.dev.view(np.uint32))
    for rr in (a, b):
        s, bits = rr.get_error()
        assert s == 0 and bits == 0


@pytest.mark.parametrize("name", list(CASES))
def test_dense_restore_equals_fused_restore(name):
    from collective_kv_cache_gb300 import runner as R
    cfg = CASES[name]
    orc = oracle.get()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg), restore=False)
    rnd = ch.rnd
    # the oracle's canonical-frame restore: X_i at agent i's positions
    pool_c = oracle.new_pool(cfg, rnd.num_pages)
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents), pool_c,
                             rnd.num_pages, rnd.block_table, frame=1) == 0

    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    a, b = _runner(cfg, rnd), _runner(cfg, rnd)
    for rr in (a, b):
        rr.rerotate(kc, vc)
        rr.check_select(R.to_device_bf16(ch.k_fresh, "cuda"))
        m = rr.pick_master()
        assert m == ch.master
        rr.alloc_store(max(rr.candidate_bound(m), 1))
        rr.diff_encode(kc, vc, R.to_device_bf16(ch.k_fresh_sel, "cuda"),
                       R.to_device_bf16(ch.v_fresh_sel, "cuda"))
        rr.pool_t.view(torch.int16).fill_(SENTINEL_I16)
    N, L, S, E = cfg.n_agents, cfg.n_layers, cfg.n_shared, cfg.elems
    a.fused_restore(list(range(N)), frame=0)
    dk = torch.empty((L, S, E), dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    for i in range(N):
        b.dense_restore([i], dk, dv)
        torch.cuda.synchronize()
        got_k, got_v = R.bits_of(dk), R.bits_of(dv)
        for l in range(L):
            assert np.array_equal(got_k[l], rk.gather_rows(pool_c, rnd.block_table, cfg.page_size,
                                                           i, l, 0, ch.pos[i])), (i, l, "K")
            assert np.array_equal(got_v[l], rk.gather_rows(pool_c, rnd.block_table, cfg.page_size,
                                                           i, l, 1, ch.pos[i])), (i, l, "V")
    assert np.array_equal(R.bits_of(a.pool_t), R.bits_of(b.pool_t))
    for rr in (a, b):
        s, bits = rr.get_error()
        assert s == 0 and bits == 0
