"""Full-size parity on the five workloads' own sizes, every layer.

The CUDA path runs the whole round at full size (all agents, layers, tokens; encode and
restore in layer chunks to bound memory). The oracle checks every layer on its own, from
inputs it builds itself with the seeded generator: the whole check layer (re-rotated rows,
deviations, selections, master and costs), and for every layer the re-rotated rows of
every agent, the recomputed inputs, the Master, every diff record of every Mirror with its
slot, and the restored rows of every agent. The oracle's recomputed inputs are its own
re-rotated rows and canonical V plus the generator's noise, which the input module draws
on the device (seed and indices in, nothing the path computed).

The oracle's work for a layer is spread over host threads (its calls release the
interpreter lock) by agent: re-rotation and restore of a group of agents write only their
own pages; a Mirror's records depend only on its own cache and the Master's, so the encode
runs on groups that each hold the Master and some Mirrors, and their records are put
back in agent order. The oracle's outputs are copied to the GPU and compared there
element by element.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

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


def _selected_noise(cfg, rnd, sel, layer, device):
    """The generator's noise for the selected tokens of one layer, [N][k][E] float32 for K
    and for V, drawn on `device` (the seeded counter-based generator of the input module:
    a function of the seed and the indices only) and returned to the host."""
    N, k, E = cfg.n_agents, sel.shape[1], cfg.elems
    nk = torch.empty((N, k, E), dtype=torch.float32, device=device)
    nv = torch.empty_like(nk)
    for i in range(N):
        tok = torch.from_numpy(sel[i].astype(np.int64)).to(device)
        pr = torch.from_numpy(rnd.perturbed[i, sel[i]]).to(device)
        nk[i] = synth.noise_rows_torch(cfg.seed, "selK", i, layer, tok, pr, E)
        nv[i] = synth.noise_rows_torch(cfg.seed, "selV", i, layer, tok, pr, E)
    return nk.cpu().numpy(), nv.cpu().numpy()


def _host_fresh_sel(cfg, rnd, pool1, pos, sel, vcl, layer, agents=None, out=None, noise=None):
    """Oracle-side recomputed K and V at the selected tokens of one layer, [N][1][k][E]:
    the oracle's own reused rows (pool1) and canonical V plus the generator's noise (the
    rows of `agents` only, into `out` when given; `noise` from _selected_noise, else drawn
    here on the host)."""
    N, k, E = cfg.n_agents, sel.shape[1], cfg.elems
    if out is None:
        out = (np.empty((N, 1, k, E), np.uint16), np.empty((N, 1, k, E), np.uint16))
    kf, vf = out
    for i in (range(N) if agents is None else agents):
        pr = rnd.perturbed[i, sel[i]]
        reused = rk.gather_rows(pool1, rnd.block_table, cfg.page_size, i, 0, 0, pos[i, sel[i]])
        if noise is None:
            nk = synth._noise_rows(cfg.seed, "selK", i, layer, sel[i], pr, E)
            nv = synth._noise_rows(cfg.seed, "selV", i, layer, sel[i], pr, E)
        else:
            nk, nv = noise[0][i], noise[1][i]
        kf[i, 0] = synth.add_noise_bf16(reused, nk)
        vf[i, 0] = synth.add_noise_bf16(vcl[0, sel[i]], nv)
    return kf, vf


WORKERS = max(2, (os.cpu_count() or 4) - 2)


def _up(a, dev):
    """A host array on the GPU (uint16 bf16 bits as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def _sub_desc(rnd, agents):
    """The round of a subset of its agents (same blocks; their histories and orders)."""
    return (rnd.block_len, rnd.hist_len[agents], np.ascontiguousarray(rnd.perm[agents]))


def _stitch(groups, results, N, m):
    """One store in agent order from encodes of agent groups that each hold the Master."""
    idx, vk, vv, counts = [], [], [], np.zeros(N, np.int64)
    where = {}
    for g, so in zip(groups, results):
        for x, i in enumerate(g):
            if i != m:
                where[i] = (so, x)
    for i in range(N):
        if i == m:
            continue
        so, x = where[i]
        a, b = int(so["rowptr"][x]), int(so["rowptr"][x + 1])
        idx.append(so["idx"][a:b])
        vk.append(so["val_k"][a:b])
        vv.append(so["val_v"][a:b])
        counts[i] = b - a
    first = results[0]
    rowptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    empty = first["val_k"][:0]
    return dict(status=0, nnz=int(rowptr[-1]), master_k=first["master_k"],
                master_v=first["master_v"], rowptr=rowptr,
                idx=np.concatenate(idx) if idx else np.zeros(0, np.int32),
                val_k=np.concatenate(vk) if vk else empty,
                val_v=np.concatenate(vv) if vv else empty)


def run_fullsize(cfg, chunk):
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import workload
    orc = oracle.get()
    dev = torch.device("cuda")
    rnd = synth.make_round(cfg)
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    N, L, S, E, P = cfg.n_agents, cfg.n_layers, cfg.n_shared, cfg.elems, cfg.page_size
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

    # ---- the check layer: deviations, selections, master and costs
    c = cfg.check_layer
    kcl, vcl = _host_canon(cfg, c)
    pool1 = oracle.new_pool(one, rnd.num_pages)
    assert orc.rerotate(one, desc, kcl, vcl, pool1, rnd.num_pages, rnd.block_table) == 0
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

    # every agent's shared rows in one layer's plane of a pool ([2][pages * P][E]), in
    # canonical token order: the same rows of the GPU pool and of an oracle pool
    bt = torch.from_numpy(np.ascontiguousarray(rnd.block_table)).to(dev).long()
    pos_t = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int64)).to(dev)
    rows_idx = (bt.gather(1, pos_t // P) * P + pos_t % P).reshape(-1)
    plane_rows = rnd.num_pages * P

    def same(gpu, host):
        return torch.equal(gpu.view(torch.int16), _up(host, dev))

    def same_rows(gpu_layer, host_pool, what, l):
        hp = _up(host_pool, dev).reshape(2, plane_rows, E)
        gp = gpu_layer.view(torch.int16).reshape(2, plane_rows, E)
        for kv in (0, 1):
            ok = torch.equal(gp[kv].index_select(0, rows_idx), hp[kv].index_select(0, rows_idx))
            assert ok, (what, l, kv)
        del hp

    # agent groups: plain partitions, and the encode's (each with the Master)
    G = min(N, WORKERS)
    parts = [np.arange(N)[g::G] for g in range(G)]
    mirrors = [i for i in range(N) if i != m_o]
    enc_groups = [np.array(sorted([m_o] + mirrors[g::G]), dtype=np.int64)
                  for g in range(min(G, max(1, len(mirrors))))]
    bt_np = rnd.block_table

    def oracle_rerotate(ex, l):
        kcl, vcl = _host_canon(cfg, l)
        p1 = oracle.new_pool(one, rnd.num_pages)
        st = list(ex.map(lambda g: orc.rerotate(one, _sub_desc(rnd, g), kcl, vcl, p1,
                                                rnd.num_pages, np.ascontiguousarray(bt_np[g])),
                         parts))
        assert all(x == 0 for x in st)
        return kcl, vcl, p1

    def oracle_encode_restore(ex, l, kcl, vcl, p1):
        k = sel_o.shape[1]
        kf_o = np.empty((N, 1, k, E), np.uint16)
        vf_o = np.empty((N, 1, k, E), np.uint16)

        noise = _selected_noise(cfg, rnd, sel_o, l, dev)
        list(ex.map(lambda g: _host_fresh_sel(cfg, rnd, p1, pos, sel_o, vcl, l, agents=g,
                                              out=(kf_o, vf_o), noise=noise), parts))
        del noise

        def enc(g):
            so = orc.diff_encode(one, _sub_desc(rnd, g), int(np.searchsorted(g, m_o)), kcl, vcl,
                                 np.ascontiguousarray(sel_o[g]), np.ascontiguousarray(kf_o[g]),
                                 np.ascontiguousarray(vf_o[g]))
            assert so["status"] == 0
            return so
        so = _stitch(enc_groups, list(ex.map(enc, enc_groups)), N, m_o)
        pr = oracle.new_pool(one, rnd.num_pages)
        st = list(ex.map(lambda g: orc.fused_restore(one, desc, m_o, so, g, pr, rnd.num_pages,
                                                     bt_np), parts))
        assert all(x == 0 for x in st)
        return kf_o, vf_o, so, pr

    total_nnz = 0
    nb = rr.nb
    with cf.ThreadPoolExecutor(WORKERS) as ex:
        for l0 in range(0, L, chunk):
            l1 = min(L, l0 + chunk)
            nl = l1 - l0
            # re-rotated rows of every layer of the chunk, before the restore rewrites them
            kept = {}
            for l in range(l0, l1):
                kcl, vcl, p1 = oracle_rerotate(ex, l)
                same_rows(rr.pool_t[l], p1, "rerotate", l)
                kept[l] = (kcl, vcl, p1)
            kfs, vfs = workload.fresh_selected(rr, rnd, sel, vc, layer_begin=l0, layer_end=l1)
            rr.alloc_store(max(int(cost_gpu[m]) * nl, 1), l0, l1)
            nnz = rr.diff_encode(kc[l0:l1], vc[l0:l1], kfs, vfs, layer_begin=l0, layer_end=l1)
            total_nnz += nnz
            rr.fused_restore(list(range(N)))
            torch.cuda.synchronize()
            t = rr.store_t
            rowptr = t["rowptr"].cpu().numpy()
            slot = t["slot"].cpu().numpy().reshape(N, nl, nb)
            for l in range(l0, l1):
                li = l - l0
                kf_o, vf_o, so, pr = oracle_encode_restore(ex, l, *kept.pop(l))
                assert same(kfs[:, li], kf_o[:, 0]), ("recomputed K", l)
                assert same(vfs[:, li], vf_o[:, 0]), ("recomputed V", l)
                assert same(t["master_k"][li], so["master_k"][0]), ("master K", l)
                assert same(t["master_v"][li], so["master_v"][0]), ("master V", l)
                # the records of layer l, Mirror by Mirror
                starts = rowptr[np.arange(N) * nl + li]
                counts = rowptr[np.arange(N) * nl + li + 1] - starts
                assert np.array_equal(counts, np.diff(so["rowptr"])), ("records", l)
                recs = np.concatenate([np.arange(a, a + n) for a, n in zip(starts, counts)]
                                      ).astype(np.int64) if counts.sum() else np.zeros(0, np.int64)
                rec_t = torch.from_numpy(recs).to(dev)
                assert np.array_equal(t["block_idx"][rec_t].cpu().numpy(), so["idx"]), \
                    ("indices", l)
                assert same(t["val_k"][rec_t], so["val_k"]), ("K values", l)
                assert same(t["val_v"][rec_t], so["val_v"]), ("V values", l)
                want = np.full((N, nb), -1, np.int64)
                for i in range(N):
                    b = so["idx"][so["rowptr"][i]:so["rowptr"][i + 1]]
                    want[i, b] = starts[i] + np.arange(len(b))
                assert np.array_equal(slot[:, li, :], want), ("slot map", l)
                same_rows(rr.pool_t[l], pr, "restore", l)
                del kf_o, vf_o, so, pr
            del kfs, vfs
            rr.store = rr.store_t = None
    s, bits = rr.get_error()
    assert s == 0 and bits == 0
    assert total_nnz > 0
    del rr, kc, vc
    torch.cuda.empty_cache()


def test_fullsize_qwen14b():
    run_fullsize(synth.qwen14b(), chunk=16)


def test_fullsize_scale64():
    run_fullsize(synth.scale64(), chunk=14)


@pytest.mark.parametrize("pct,page", [(5, 16), (10, 32), (20, 16), (40, 32), (40, 16)])
def test_fullsize_density(pct, page):
    """Recompute fractions 5-40% in clustered runs; pages 16 and 32, block tables permuted
    across a 120 GB pool."""
    run_fullsize(synth.density(pct, page_size=page), chunk=8)
