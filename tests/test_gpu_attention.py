"""Decode attention read from the Master and the diffs (td_fused_attention), and the same
attention over a restored cache (td_paged_attention), against the float64 oracle.

Tolerance, from the kernels' arithmetic (per output element of query head g of agent a):
a shared block's query is turned in float32 and split into two bf16 parts (the residual is
at most 2^-16 |q| per element), the products are exact and the tensor cores accumulate in
float32 over 2D/16 chunks, so a score is off by at most
    delta = scale * 2^-15 * |q| * max_p |k_p|           (Cauchy-Schwarz on sum |q_d k_pd|);
softmax weights then move by at most 2 delta (relative), and float32 sums over at most
512 positions per unit and a few dozen units add 2^-13 relative. Hence
    |out - out64| <= max_p |v_p| * (2 delta + 2^-13)   and   |lse - lse64| <= delta + 2^-13.
A history query is bf16 already, so the same bound holds with room to spare.
"""
from __future__ import annotations

import math

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
    base = dict(name="mini", n_agents=4, n_layers=2, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(3, 45), check_layer=1,
                recompute_pct=15, perturb_mode="runs", perturb_frac=(0.10, 0.20), seed=101)
    base.update(kw)
    return synth.RoundConfig(**base)


CASES = {
    "mini_gqa3": (_mini(), 6),
    "mini_d128_gqa2": (_mini(head_dim=128, seed=102), 4),
    "mini_no_gqa": (_mini(seed=103), 2),
    "mini_gqa8": (_mini(seed=104), 16),
    "mini_b32_p32": (_mini(diff_block=32, page_size=32, seed=105), 6),
    "mini_one_agent": (_mini(n_agents=1, seed=106), 6),
    "mini_no_history": (_mini(hist_range=(0, 0), seed=107), 6),
    "mini_long_history": (_mini(hist_range=(700, 1500), seed=108), 6),   # several units each
    "mini_pct100": (_mini(recompute_pct=100, seed=109), 6),
    # pages that do not hold a whole stage: a box reaches past the stage's page
    "mini_p24": (_mini(page_size=24, hist_range=(30, 100), seed=115), 6),
    "mini_p8_d128": (_mini(page_size=8, head_dim=128, hist_range=(30, 100), seed=116), 4),
    "qwen7b_2layers": (synth.qwen7b().replace(n_layers=2), 28),
    # more than one wave of 512-position units on a 152-SM GPU (13 a SM) while a layer is
    # under half a wave: the grid ends with the last 4 of the 8 layers in 128-position units
    "wide_p24": (_mini(n_agents=16, n_layers=8, page_size=24, hist_range=(3000, 5000),
                       seed=117), 6),
    "wide_b32_p32": (_mini(n_agents=16, n_layers=8, diff_block=32, page_size=32,
                           hist_range=(3000, 5000), seed=118), 6),
}


def _store_tensors(cfg, store, dev):
    """The oracle's store on the device, with the slot map its CSR rows imply."""
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    N, L, S, B, E = cfg.n_agents, cfg.n_layers, cfg.n_shared, cfg.diff_block, cfg.elems
    nb = (S + B - 1) // B
    slot = np.full(N * L * nb, -1, dtype=np.int32)
    for row in range(N * L):
        for r in range(store["rowptr"][row], store["rowptr"][row + 1]):
            slot[row * nb + store["idx"][r]] = r
    nnz = store["nnz"]
    t = dict(master_k=R.to_device_bf16(store["master_k"], dev),
             master_v=R.to_device_bf16(store["master_v"], dev),
             rowptr=torch.from_numpy(store["rowptr"]).to(dev),
             block_idx=torch.from_numpy(np.maximum(store["idx"], 0).astype(np.int32)
                                        if nnz else np.zeros(1, np.int32)).to(dev),
             val_k=R.to_device_bf16(store["val_k"] if nnz else np.zeros((1, B, E), np.uint16), dev),
             val_v=R.to_device_bf16(store["val_v"] if nnz else np.zeros((1, B, E), np.uint16), dev),
             slot=torch.from_numpy(slot).to(dev))
    st = td.make_store(t["master_k"], t["master_v"], t["rowptr"], t["block_idx"], t["val_k"],
                       t["val_v"], t["slot"])
    st.layer_begin, st.layer_end = 0, L
    return t, st


def _bounds(cfg, q, ctx_k_norm, vmax, scale, restored=False):
    """Per (layer, agent, query head) tolerance of the output and of the log-sum-exp."""
    qf = synth.bf16_bits_to_f32(q).astype(np.float64)
    qn = np.linalg.norm(qf, axis=-1)                          # [nl][n][nq]
    rel = 2.0 ** -15 + (2.0 ** -8 if restored else 0.0)
    delta = scale * rel * qn * ctx_k_norm
    return vmax * (2 * delta + 2.0 ** -13) + 1e-6, delta + 2.0 ** -13 + 1e-6


def _context_stats(cfg, ch, pool, nq):
    """max_p |k_p| (exact turned keys) and max_p |v_p| per (layer, agent, query head)."""
    orc = oracle.get()
    rnd, H, D, P = ch.rnd, cfg.n_kv_heads, cfg.head_dim, cfg.page_size
    N, L = cfg.n_agents, cfg.n_layers
    G = nq // H
    kn = np.zeros((L, N, nq))
    vm = np.zeros((L, N, nq))
    pool_c = oracle.new_pool(cfg, rnd.num_pages)
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(N), pool_c,
                             rnd.num_pages, rnd.block_table, frame=1) == 0
    for a in range(N):
        h = int(rnd.hist_len[a])
        for l in range(L):
            hk = synth.bf16_bits_to_f32(rk.gather_rows(pool, rnd.block_table, P, a, l, 0, np.arange(h)))
            hv = synth.bf16_bits_to_f32(rk.gather_rows(pool, rnd.block_table, P, a, l, 1, np.arange(h)))
            sx = synth.bf16_bits_to_f32(rk.gather_rows(pool_c, rnd.block_table, P, a, l, 0, ch.pos[a]))
            sv = synth.bf16_bits_to_f32(rk.gather_rows(pool_c, rnd.block_table, P, a, l, 1, ch.pos[a]))
            K = np.concatenate([hk, sx]).reshape(-1, H, D)       # rotation keeps norms
            V = np.concatenate([hv, sv]).reshape(-1, H, D)
            kmax = np.linalg.norm(K.astype(np.float64), axis=-1).max(axis=0)   # [H]
            vmax = np.abs(V).max(axis=(0, 2))
            kn[l, a] = np.repeat(kmax, G) * (1 + 2.0 ** -7)     # bf16 of a turned key
            vm[l, a] = np.repeat(vmax, G)
    return kn, vm


def _run(name, paged):
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg, nq = CASES[name]
    orc = oracle.get()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, map_history=True), restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages, fill=0x7FC0)     # NaN where nothing belongs
    rk.fill_history(cfg, rnd, pool)
    if paged:
        assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents), pool,
                                 rnd.num_pages, rnd.block_table, frame=0) == 0
    agents = list(range(cfg.n_agents))
    q = synth.decode_queries(cfg, nq, agents, 0, cfg.n_layers)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    st, out_o, lse_o = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool,
                                     rnd.num_pages, rnd.block_table, q, nq, scale, from_pool=paged)
    assert st == 0

    dev = torch.device("cuda")
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages)
    rr.pool_t.copy_(R.to_device_bf16(pool, dev).reshape(rr.pool_t.shape))
    qd = R.to_device_bf16(q, dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device=dev)
    if paged:
        td.td_paged_attention(rr.ctx.handle, rr.round, rr.pool, agents, 0, cfg.n_layers,
                              qd.data_ptr(), nq, scale, out.data_ptr(), lse.data_ptr(), rr.s)
    else:
        _, store = _store_tensors(cfg, ch.store, dev)
        td.td_fused_attention(rr.ctx.handle, rr.round, store, rr.pool, agents, 0, cfg.n_layers,
                              qd.data_ptr(), nq, scale, out.data_ptr(), lse.data_ptr(), rr.s)
    torch.cuda.synchronize()
    s, bits = rr.get_error()
    assert s == 0 and bits == 0, (s, bits)
    got, got_lse = out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all() and np.isfinite(got_lse).all()
    kn, vm = _context_stats(cfg, ch, pool, nq)
    tol, tol_lse = _bounds(cfg, q, kn, vm, scale)
    err = np.abs(got - out_o).max(axis=-1)
    assert (err <= tol).all(), (float(err.max()), float(tol.min()))
    assert (np.abs(got_lse - lse_o) <= tol_lse).all()
    return float(err.max())


@pytest.mark.parametrize("name", list(CASES))
def test_fused_attention_matches_oracle(name):
    _run(name, paged=False)


@pytest.mark.parametrize("name", ["mini_gqa3", "mini_d128_gqa2", "mini_long_history",
                                  "qwen7b_2layers", "wide_p24"])
def test_paged_attention_matches_oracle(name):
    _run(name, paged=True)


def test_fused_attention_agent_subset_and_layer_range():
    """A subset of agents in any order and a layer sub-range give the same rows."""
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg, nq = _mini(n_layers=3, n_agents=5, seed=110), 6
    orc = oracle.get()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, map_history=True), restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages)
    rk.fill_history(cfg, rnd, pool)
    agents = [4, 1, 3]
    q = synth.decode_queries(cfg, nq, agents, 1, 3)
    scale = 0.2
    # the oracle's store for layers 1..2 alone
    kf, vf = ch.k_fresh_sel[:, 1:3].copy(), ch.v_fresh_sel[:, 1:3].copy()
    store12 = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel, kf, vf, 1, 3)
    assert store12["status"] == 0
    sub = cfg.replace(n_layers=3)
    st, out_o, _ = orc.attention(sub, ch.desc, ch.master, store12, agents, pool, rnd.num_pages,
                                 rnd.block_table, q, nq, scale, layer_begin=1, layer_end=3)
    assert st == 0
    dev = torch.device("cuda")
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table, rnd.num_pages)
    rr.pool_t.copy_(R.to_device_bf16(pool, dev).reshape(rr.pool_t.shape))
    t, store = _store_tensors(cfg.replace(n_layers=2), store12, dev)
    store.layer_begin, store.layer_end = 1, 3
    qd = R.to_device_bf16(q, dev)
    out = torch.zeros(q.shape, dtype=torch.float32, device=dev)
    td.td_fused_attention(rr.ctx.handle, rr.round, store, rr.pool, agents, 1, 3, qd.data_ptr(),
                          nq, scale, out.data_ptr(), None, rr.s)
    torch.cuda.synchronize()
    assert rr.get_error()[0] == 0
    # the derived bound is about 5e-3 here; a wrong row or rotation moves outputs by ~0.1
    assert np.abs(out.cpu().numpy() - out_o).max() < 5e-3


def test_fused_attention_rejects_bad_arguments():
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg = _mini(seed=111)
    rnd = synth.make_round(cfg, map_history=True)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table, rnd.num_pages)
    rr.alloc_store(4)
    rr.store.layer_begin, rr.store.layer_end = 0, cfg.n_layers
    q = torch.zeros((cfg.n_layers, 1, 6, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    bad = [dict(nq=5), dict(nq=2 * 9), dict(agents=[cfg.n_agents]), dict(lb=1, le=1),
           dict(lb=0, le=cfg.n_layers + 1)]
    for b in bad:
        with pytest.raises(td.TDError):
            td.td_fused_attention(rr.ctx.handle, rr.round, rr.store, rr.pool, b.get("agents", [0]),
                                  b.get("lb", 0), b.get("le", cfg.n_layers), q.data_ptr(),
                                  b.get("nq", 6), 0.1, out.data_ptr(), None, rr.s)
    # no agents: nothing to do
    td.td_fused_attention(rr.ctx.handle, rr.round, rr.store, rr.pool, [], 0, cfg.n_layers,
                          q.data_ptr(), 6, 0.1, out.data_ptr(), None, rr.s)


def test_wait_timeout_is_reported_and_the_context_recovers():
    """Fault injection on the host (td_inject_attention_wait_fault): every stage's barrier
    expects bytes that never come, each bounded wait runs out, the error word says
    TD_ERR_DEVICE_TIMEOUT and nothing faults; the next call on the same context is right."""
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg, nq = _mini(n_agents=2, n_layers=1, check_layer=0, seed=112), 6
    orc = oracle.get()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, map_history=True), restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages)
    rk.fill_history(cfg, rnd, pool)
    agents = list(range(cfg.n_agents))
    q = synth.decode_queries(cfg, nq, agents, 0, 1)
    st, out_o, _ = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool, rnd.num_pages,
                                 rnd.block_table, q, nq, 0.125)
    assert st == 0
    dev = torch.device("cuda")
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table, rnd.num_pages)
    rr.pool_t.copy_(R.to_device_bf16(pool, dev).reshape(rr.pool_t.shape))
    _, store = _store_tensors(cfg, ch.store, dev)
    qd = R.to_device_bf16(q, dev)
    out = torch.zeros(q.shape, dtype=torch.float32, device=dev)

    def call():
        td.td_fused_attention(rr.ctx.handle, rr.round, store, rr.pool, agents, 0, 1,
                              qd.data_ptr(), nq, 0.125, out.data_ptr(), None, rr.s)

    td.td_inject_attention_wait_fault(rr.ctx.handle, 16)
    call()
    s, bits = rr.get_error()
    assert s == td.TD_ERR_DEVICE_TIMEOUT and bits == (1 << td.TD_ERR_DEVICE_TIMEOUT), (s, bits)
    td.td_inject_attention_wait_fault(rr.ctx.handle, 0)
    call()
    s, bits = rr.get_error()
    assert s == 0 and bits == 0
    assert np.abs(out.cpu().numpy() - out_o).max() < 5e-3


def test_fused_attention_refuses_a_store_in_host_memory():
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    import bench
    cfg = _mini(seed=113)
    rnd = synth.make_round(cfg, map_history=True)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table, rnd.num_pages)
    bench.host_store(rr, 8)
    rr.store.layer_begin, rr.store.layer_end = 0, cfg.n_layers
    q = torch.zeros((cfg.n_layers, 1, 6, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(td.TDError):
        td.td_fused_attention(rr.ctx.handle, rr.round, rr.store, rr.pool, [0], 0, cfg.n_layers,
                              q.data_ptr(), 6, 0.1, out.data_ptr(), None, rr.s)


def test_three_hundred_agents_span_two_launches():
    """More agents than one launch carries (256): restore and both attentions split the
    list; every agent's rows must still be right, the second launch's included."""
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import td
    cfg = _mini(n_agents=300, n_layers=1, check_layer=0, block_lens=(20, 13), hist_range=(0, 20),
                seed=114)
    nq = 4
    orc = oracle.get()
    ch = rk.run_oracle_chain(rk.make_inputs(cfg, map_history=True), restore=False)
    rnd = ch.rnd
    pool = oracle.new_pool(cfg, rnd.num_pages)
    rk.fill_history(cfg, rnd, pool)
    agents = list(range(cfg.n_agents))[::-1]            # reversed, so list order matters
    q = synth.decode_queries(cfg, nq, agents, 0, 1)
    st, out_o, lse_o = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool,
                                     rnd.num_pages, rnd.block_table, q, nq, 0.125)
    assert st == 0
    dev = torch.device("cuda")
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table, rnd.num_pages)
    rr.pool_t.copy_(R.to_device_bf16(pool, dev).reshape(rr.pool_t.shape))
    t, store = _store_tensors(cfg, ch.store, dev)
    qd = R.to_device_bf16(q, dev)
    out = torch.zeros(q.shape, dtype=torch.float32, device=dev)
    lse = torch.zeros(q.shape[:-1], dtype=torch.float32, device=dev)
    td.td_fused_attention(rr.ctx.handle, rr.round, store, rr.pool, agents, 0, 1, qd.data_ptr(),
                          nq, 0.125, out.data_ptr(), lse.data_ptr(), rr.s)
    torch.cuda.synchronize()
    assert rr.get_error()[0] == 0
    assert np.abs(out.cpu().numpy() - out_o).max() < 5e-3
    assert np.abs(lse.cpu().numpy() - lse_o).max() < 5e-3
    # the restore over the same 300 agents, bit for bit, then attention over the pages
    pool_r = pool.copy()
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.asarray(agents), pool_r,
                             rnd.num_pages, rnd.block_table, frame=0) == 0
    rr.store = store
    store.layer_begin, store.layer_end = 0, 1
    rr.fused_restore(agents)
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(rr.pool_t), pool_r)
    st, out_p, _ = orc.attention(cfg, ch.desc, ch.master, ch.store, agents, pool_r,
                                 rnd.num_pages, rnd.block_table, q, nq, 0.125, from_pool=True)
    assert st == 0
    td.td_paged_attention(rr.ctx.handle, rr.round, rr.pool, agents, 0, 1, qd.data_ptr(), nq,
                          0.125, out.data_ptr(), None, rr.s)
    torch.cuda.synchronize()
    assert rr.get_error()[0] == 0
    assert np.abs(out.cpu().numpy() - out_p).max() < 5e-3
