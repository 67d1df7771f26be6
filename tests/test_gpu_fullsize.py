"""Full-size parity on the five workloads' own sizes.

The CUDA path runs the whole round at full size (all agents, layers, tokens; encode and
restore in layer chunks to bound memory). The oracle cannot hold a full-size round, so it
checks what it can compute on its own: the whole check layer (re-rotated rows, deviations,
selections, master and costs) and a few sampled layers (re-rotated rows, the recomputed
inputs, every diff record of every Mirror, the Master, and the restored rows of every
agent), each from inputs it builds itself with the seeded generator.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_kv_cache_gb300 import synth
from tests import roundkit as rk

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()
    torch.set_num_threads(max(1, torch.get_num_threads()))


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _host_canon(cfg, layer):
    k = synth.canonical_torch(cfg, "K", layer, "cpu")
    v = synth.canonical_torch(cfg, "V", layer, "cpu")
    return _bits(k)[None], _bits(v)[None]


def _host_fresh_check(cfg, rnd, pool1, pos):
    """Oracle-side recomputed K at the check layer (from its own one-layer pool)."""
    out = np.empty((cfg.n_agents, cfg.n_shared, cfg.elems), np.uint16)
    tok = torch.arange(cfg.n_shared, dtype=torch.int64)
    for i in range(cfg.n_agents):
        reused = rk.gather_rows(pool1, rnd.block_table, cfg.page_size, i, 0, 0, pos[i])
        noise = synth.noise_rows_torch(cfg.seed, "chk", i, cfg.check_layer, tok,
                                       torch.from_numpy(rnd.perturbed[i]), cfg.elems).numpy()
        out[i] = synth.add_noise_bf16(reused, noise)
    return out


def _host_fresh_sel(cfg, rnd, pool1, pos, sel, vcl, layer):
    N, k, E = cfg.n_agents, sel.shape[1], cfg.elems
    kf = np.empty((N, 1, k, E), np.uint16)
    vf = np.empty((N, 1, k, E), np.uint16)
    for i in range(N):
        tok = torch.from_numpy(sel[i].astype(np.int64))
        pr = torch.from_numpy(rnd.perturbed[i, sel[i]])
        reused = rk.gather_rows(pool1, rnd.block_table, cfg.page_size, i, 0, 0, pos[i, sel[i]])
        nk = synth.noise_rows_torch(cfg.seed, "selK", i, layer, tok, pr, E).numpy()
        nv = synth.noise_rows_torch(cfg.seed, "selV", i, layer, tok, pr, E).numpy()
        kf[i, 0] = synth.add_noise_bf16(reused, nk)
        vf[i, 0] = synth.add_noise_bf16(vcl[0, sel[i]], nv)
    return kf, vf


def _agent_rows_gpu(rr, layer, kv, pos):
    return np.stack([_bits(rr.gather(i, layer, kv, pos[i])) for i in range(rr.N)])


def _agent_rows_host(cfg, rnd, pool1, kv, pos):
    return np.stack([rk.gather_rows(pool1, rnd.block_table, cfg.page_size, i, 0, kv, pos[i])
                     for i in range(cfg.n_agents)])


def run_fullsize(cfg, sample_layers, chunk):
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import workload
    orc = oracle.get()
    dev = torch.device("cuda")
    rnd = synth.make_round(cfg)
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    N, L, S = cfg.n_agents, cfg.n_layers, cfg.n_shared
    one = cfg.replace(n_layers=1, check_layer=0)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, device=dev)
    pos = rr.positions()
    kc, vc = workload.canonical(cfg, dev)
    rr.rerotate(kc, vc)
    kf = workload.fresh_check(rr, rnd)
    sel_t = rr.check_select(kf)
    m = rr.pick_master()
    sel = sel_t.cpu().numpy()
    dev_gpu = rr.dev_t.cpu().numpy()
    cost_gpu = rr.cost_t.cpu().numpy()

    # ---- the check layer, whole
    c = cfg.check_layer
    kcl, vcl = _host_canon(cfg, c)
    pool1 = oracle.new_pool(one, rnd.num_pages)
    assert orc.rerotate(one, desc, kcl, vcl, pool1, rnd.num_pages, rnd.block_table) == 0
    for kv in (0, 1):
        assert np.array_equal(_agent_rows_gpu(rr, c, kv, pos),
                              _agent_rows_host(cfg, rnd, pool1, kv, pos)), ("rerotate", c, kv)
    kf_o = _host_fresh_check(cfg, rnd, pool1, pos)
    assert np.array_equal(_bits(kf), kf_o), "recomputed K at the check layer"
    st, sel_o, dev_o = orc.check_select(one, desc, pool1, rnd.num_pages, rnd.block_table, kf_o,
                                        check_layer=0, pct=cfg.recompute_pct)
    assert st == 0
    assert np.array_equal(dev_gpu.view(np.uint32), dev_o.view(np.uint32)), "deviations"
    assert np.array_equal(sel, sel_o), "selections"
    m_o, cost_o = orc.pick_master(S, cfg.diff_block, sel_o)
    assert m == m_o and np.array_equal(cost_gpu, cost_o), (m, m_o)
    del pool1, kf_o, kf

    # ---- all layers in chunks on the GPU; sampled layers against the oracle
    total_nnz = 0
    for l0 in range(0, L, chunk):
        l1 = min(L, l0 + chunk)
        in_chunk = [l for l in sample_layers if l0 <= l < l1]
        refs = {}
        for l in in_chunk:                       # re-rotated rows, before restore rewrites them
            kcl, vcl = _host_canon(cfg, l)
            p1 = oracle.new_pool(one, rnd.num_pages)
            assert orc.rerotate(one, desc, kcl, vcl, p1, rnd.num_pages, rnd.block_table) == 0
            for kv in (0, 1):
                assert np.array_equal(_agent_rows_gpu(rr, l, kv, pos),
                                      _agent_rows_host(cfg, rnd, p1, kv, pos)), ("rerotate", l, kv)
            refs[l] = (kcl, vcl, p1)
        kfs, vfs = workload.fresh_selected(rr, rnd, sel, vc, layer_begin=l0, layer_end=l1)
        rr.alloc_store(max(int(cost_gpu[m]) * (l1 - l0), 1), l0, l1)
        nnz = rr.diff_encode(kc[l0:l1], vc[l0:l1], kfs, vfs, layer_begin=l0, layer_end=l1)
        total_nnz += nnz
        rr.fused_restore(list(range(N)))
        torch.cuda.synchronize()
        t = rr.store_t
        rowptr = t["rowptr"].cpu().numpy()
        for l, (kcl, vcl, p1) in refs.items():
            li = l - l0
            kf_o, vf_o = _host_fresh_sel(cfg, rnd, p1, pos, sel_o, vcl, l)
            assert np.array_equal(_bits(kfs[:, li]), kf_o[:, 0]), ("recomputed K", l)
            assert np.array_equal(_bits(vfs[:, li]), vf_o[:, 0]), ("recomputed V", l)
            so = orc.diff_encode(one, desc, m_o, kcl, vcl, sel_o, kf_o, vf_o)
            assert so["status"] == 0
            assert np.array_equal(_bits(t["master_k"][li]), so["master_k"][0]), ("master K", l)
            assert np.array_equal(_bits(t["master_v"][li]), so["master_v"][0]), ("master V", l)
            for i in range(N):
                r = i * (l1 - l0) + li
                a0, a1 = int(rowptr[r]), int(rowptr[r + 1])
                b0, b1 = int(so["rowptr"][i]), int(so["rowptr"][i + 1])
                assert a1 - a0 == b1 - b0, ("records", l, i)
                assert np.array_equal(t["block_idx"][a0:a1].cpu().numpy(), so["idx"][b0:b1])
                assert np.array_equal(_bits(t["val_k"][a0:a1]), so["val_k"][b0:b1]), ("K", l, i)
                assert np.array_equal(_bits(t["val_v"][a0:a1]), so["val_v"][b0:b1]), ("V", l, i)
            pr = oracle.new_pool(one, rnd.num_pages)
            assert orc.fused_restore(one, desc, m_o, so, np.arange(N), pr, rnd.num_pages,
                                     rnd.block_table) == 0
            for kv in (0, 1):
                assert np.array_equal(_agent_rows_gpu(rr, l, kv, pos),
                                      _agent_rows_host(cfg, rnd, pr, kv, pos)), ("restore", l, kv)
            del pr, so, kf_o, vf_o
        del kfs, vfs, refs
        rr.store = rr.store_t = None
    s, bits = rr.get_error()
    assert s == 0 and bits == 0
    assert total_nnz > 0
    del rr, kc, vc
    torch.cuda.empty_cache()


def test_fullsize_qwen14b():
    cfg = synth.qwen14b()
    run_fullsize(cfg, sample_layers=[1, 26, 47], chunk=16)


def test_fullsize_scale64():
    cfg = synth.scale64()
    run_fullsize(cfg, sample_layers=[1, 27], chunk=14)


@pytest.mark.parametrize("pct,page", [(5, 16), (10, 32), (20, 16), (40, 32), (40, 16)])
def test_fullsize_density(pct, page):
    """Recompute fractions 5-40% in clustered runs; pages 16 and 32, block tables permuted
    across a 120 GB pool."""
    cfg = synth.density(pct, page_size=page)
    run_fullsize(cfg, sample_layers=[1, 40], chunk=8)
