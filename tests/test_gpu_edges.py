"""Edge cases of the CUDA path against the oracle: compaction when candidate blocks equal
the Master's, undersized stores, unmapped pages, non-finite deviations, invalid arguments,
layer sub-ranges and partial agent lists. No case faults the GPU: every fault is made on
the host (tables, sizes, inputs) and is caught by host validation or the device error
word."""
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


def _R():
    from collective_kv_cache_gb300 import runner as R
    return R


def _mini(**kw):
    base = dict(name="mini", n_agents=3, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(0, 0), hist_fixed=(7, 7, 30),
                check_layer=1, recompute_pct=15, seed=91)
    base.update(kw)
    return synth.RoundConfig(**base)


def _twin_inputs():
    """Agents 0 and 1 share placement, selection and recomputed values (so every
    candidate block of Mirror 1 equals the Master's), agent 2 differs."""
    cfg = _mini()
    ch = rk.make_inputs(cfg)
    ch.rnd.perm[1] = ch.rnd.perm[0]
    ch.off = oracle.get().offsets(*ch.desc)
    ch.pos = rk.positions(ch.off, ch.rnd.block_len)
    rng = np.random.default_rng(5)
    S, L, E = cfg.n_shared, cfg.n_layers, cfg.elems
    k = 9
    s01 = np.sort(rng.choice(S, k, replace=False)).astype(np.int32)
    s2 = np.sort(rng.choice(S, k, replace=False)).astype(np.int32)
    sel = np.stack([s01, s01, s2])
    vals = synth.f32_to_bf16_bits(rng.standard_normal((3, L, k, E)).astype(np.float32))
    vals[1] = vals[0]
    vv = synth.f32_to_bf16_bits(rng.standard_normal((3, L, k, E)).astype(np.float32))
    vv[1] = vv[0]
    return cfg, ch, sel, vals, vv


def _runner(cfg, ch, fill=None):
    R = _R()
    return R.RoundRunner(cfg, ch.rnd.block_len, ch.rnd.hist_len, ch.rnd.perm,
                         ch.rnd.block_table, ch.rnd.num_pages, pool_fill=fill)


def test_encode_compacts_when_candidates_equal_the_master():
    R = _R()
    cfg, ch, sel, kf, vf = _twin_inputs()
    orc = oracle.get()
    want = orc.diff_encode(cfg, ch.desc, 0, ch.kc, ch.vc, sel, kf, vf)
    assert want["status"] == 0
    rows = np.diff(want["rowptr"]).reshape(3, cfg.n_layers)
    assert rows[1].sum() == 0 and rows[2].sum() > 0      # Mirror 1 needs no record
    rr = _runner(cfg, ch)
    m, _ = orc.pick_master(cfg.n_shared, 16, sel)
    sel_t = torch.from_numpy(sel).cuda()
    rr.pick_master(sel_t)
    rr.master_t.fill_(0)                                # the caller's own choice
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    bound = int(rr.cost_t[0].item()) * cfg.n_layers
    assert bound > want["nnz"]
    rr.alloc_store(bound)
    nnz = rr.diff_encode(kc, vc, R.to_device_bf16(kf, "cuda"), R.to_device_bf16(vf, "cuda"),
                         sel=sel_t)
    assert nnz == want["nnz"]
    t = rr.store_t
    assert np.array_equal(t["rowptr"].cpu().numpy(), want["rowptr"])
    assert np.array_equal(t["block_idx"].cpu().numpy()[:nnz], want["idx"])
    assert np.array_equal(R.bits_of(t["val_k"][:nnz]), want["val_k"])
    assert np.array_equal(R.bits_of(t["val_v"][:nnz]), want["val_v"])
    assert np.array_equal(R.bits_of(t["master_k"]), want["master_k"])
    slot = t["slot"].cpu().numpy().reshape(3, cfg.n_layers, rr.nb)
    assert (slot[0] == -1).all() and (slot[1] == -1).all()
    # restore (canonical frame) of every agent gives back its own cache
    pool_o = oracle.new_pool(cfg, ch.rnd.num_pages)
    assert orc.fused_restore(cfg, ch.desc, 0, want, np.arange(3), pool_o, ch.rnd.num_pages,
                             ch.rnd.block_table, frame=1) == 0
    rr.pool_t.zero_()
    rr.fused_restore([0, 1, 2], frame=1)
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(rr.pool_t), pool_o)
    s, bits = rr.get_error()
    assert s == 0 and bits == 0


def test_encode_capacity_error_writes_no_values():
    R = _R()
    cfg, ch, sel, kf, vf = _twin_inputs()
    rr = _runner(cfg, ch)
    sel_t = torch.from_numpy(sel).cuda()
    rr.pick_master(sel_t)
    bound = int(rr.cost_t[rr.master_t.item()].item()) * cfg.n_layers
    rr.alloc_store(bound - 1)
    rr.store_t["val_k"].view(torch.int16).fill_(0x1234)
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    s, nnz = rr.diff_encode(kc, vc, R.to_device_bf16(kf, "cuda"), R.to_device_bf16(vf, "cuda"),
                            sel=sel_t, check=False)
    from collective_kv_cache_gb300 import td
    assert s == td.TD_ERR_CAPACITY and nnz == bound
    assert (rr.store_t["val_k"].view(torch.int16) == 0x1234).all()
    st, bits = rr.get_error()
    assert bits & (1 << td.TD_ERR_CAPACITY)


def test_unmapped_page_is_reported_and_skipped():
    R = _R()
    from collective_kv_cache_gb300 import td
    cfg = _mini(hist_fixed=(7, 7, 30))
    ch = rk.make_inputs(cfg)
    bt = ch.rnd.block_table.copy()
    lp = int(ch.pos[2, 5]) // cfg.page_size
    bt[2, lp] = -1                                       # a page of agent 2's shared span
    orc = oracle.get()
    pool_o = oracle.new_pool(cfg, ch.rnd.num_pages, fill=0x5555)
    st = orc.rerotate(cfg, ch.desc, ch.kc, ch.vc, pool_o, ch.rnd.num_pages, bt)
    assert st == oracle.ORC_ERR_UNMAPPED
    rr = R.RoundRunner(cfg, ch.rnd.block_len, ch.rnd.hist_len, ch.rnd.perm, bt,
                       ch.rnd.num_pages, pool_fill=0x5555)
    rr.rerotate(R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda"))
    s, bits = rr.get_error()
    assert s == td.TD_ERR_UNMAPPED_PAGE
    assert np.array_equal(R.bits_of(rr.pool_t), pool_o)
    s, bits = rr.get_error()                             # the word was cleared
    assert s == 0 and bits == 0


def test_nonfinite_deviation_is_reported():
    R = _R()
    from collective_kv_cache_gb300 import td
    cfg = _mini()
    ch = rk.make_inputs(cfg)
    rr = _runner(cfg, ch)
    rr.rerotate(R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda"))
    kf = np.zeros((cfg.n_agents, cfg.n_shared, cfg.elems), np.uint16)
    kf[1, 3, 17] = 0x7FC0                                # NaN in one recomputed key
    rr.check_select(R.to_device_bf16(kf, "cuda"))
    s, bits = rr.get_error()
    assert s == td.TD_ERR_NONFINITE


def test_invalid_arguments_are_rejected_before_launch():
    R = _R()
    from collective_kv_cache_gb300 import td
    cfg = _mini()
    ch = rk.make_inputs(cfg)
    rr = _runner(cfg, ch)
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    h = rr.ctx.handle
    assert td.td_rerotate_batched(h, rr.round, kc.data_ptr(), vc.data_ptr(), 0, cfg.n_layers + 1,
                                  rr.pool, check=False) == td.TD_ERR_INVALID_ARG
    assert td.td_rerotate_batched(h, rr.round, None, vc.data_ptr(), 0, 1, rr.pool,
                                  check=False) == td.TD_ERR_INVALID_ARG
    assert td.td_rerotate_batched(h, rr.round, kc.data_ptr() + 2, None, 0, 1, rr.pool,
                                  check=False) == td.TD_ERR_INVALID_ARG      # misaligned
    bad = td.make_round(ch.rnd.block_len, ch.rnd.hist_len, np.zeros_like(ch.rnd.perm))
    assert td.td_rerotate_batched(h, bad, kc.data_ptr(), None, 0, 1, rr.pool,
                                  check=False) == td.TD_ERR_INVALID_ARG      # not a permutation
    short = td.make_paged(rr.pool_t, rr.bt_t[:, :1].contiguous())
    assert td.td_rerotate_batched(h, rr.round, kc.data_ptr(), None, 0, 1, short,
                                  check=False) == td.TD_ERR_INVALID_ARG      # table too short
    s, _ = td.td_check_select(h, rr.round, 0, rr.pool, kc.data_ptr(), 101, None, check=False)
    assert s == td.TD_ERR_INVALID_ARG
    s, bits = rr.get_error()
    assert s == 0 and bits == 0                         # nothing ran


def test_layer_subrange_and_agent_subset():
    """Encode layers [1, 3) only and restore layer 2 of agents [2, 0]: compare with the
    oracle on the same sub-range; other agents' and layers' rows stay untouched."""
    R = _R()
    cfg = _mini(n_agents=4, hist_fixed=(3, 40, 0, 17))
    ch = rk.run_oracle_chain(rk.make_inputs(cfg), restore=False)
    orc = oracle.get()
    lb, le = 1, 3
    want = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel,
                           np.ascontiguousarray(ch.k_fresh_sel[:, lb:le]),
                           np.ascontiguousarray(ch.v_fresh_sel[:, lb:le]), lb, le)
    rr = _runner(cfg, ch, fill=0x1111)
    sel_t = torch.from_numpy(ch.sel).cuda()
    m = rr.pick_master(sel_t)
    assert m == ch.master
    rr.alloc_store(max(rr.candidate_bound(m, lb, le), 1), lb, le)
    kc = R.to_device_bf16(np.ascontiguousarray(ch.kc[lb:le]), "cuda")
    vc = R.to_device_bf16(np.ascontiguousarray(ch.vc[lb:le]), "cuda")
    nnz = rr.diff_encode(kc, vc, R.to_device_bf16(np.ascontiguousarray(ch.k_fresh_sel[:, lb:le]), "cuda"),
                         R.to_device_bf16(np.ascontiguousarray(ch.v_fresh_sel[:, lb:le]), "cuda"),
                         sel=sel_t, layer_begin=lb, layer_end=le)
    assert nnz == want["nnz"]
    assert np.array_equal(rr.store_t["rowptr"].cpu().numpy(), want["rowptr"])
    assert np.array_equal(R.bits_of(rr.store_t["val_k"][:nnz]), want["val_k"])
    # encoding is per layer, so the oracle's store of layer 2 alone holds the same records
    want2 = orc.diff_encode(cfg, ch.desc, ch.master, ch.kc, ch.vc, ch.sel,
                            np.ascontiguousarray(ch.k_fresh_sel[:, 2:3]),
                            np.ascontiguousarray(ch.v_fresh_sel[:, 2:3]), 2, 3)
    pool_o = oracle.new_pool(cfg, ch.rnd.num_pages, fill=0x1111)
    assert orc.fused_restore(cfg, ch.desc, ch.master, want2, np.array([2, 0]), pool_o,
                             ch.rnd.num_pages, ch.rnd.block_table, layer_begin=2, layer_end=3) == 0
    rr.fused_restore([2, 0], layer_begin=2, layer_end=3)
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(rr.pool_t), pool_o)


def test_overlapped_round_matches_oracle():
    """Selection, master and encode on a second stream, overlapped with the re-rotation of
    the other layers: the store and the restored pool are still the oracle's, bit for
    bit."""
    R = _R()
    cfg = synth.qwen7b().replace(n_layers=4, check_layer=2)
    ch = rk.run_oracle_chain(rk.make_inputs(cfg))
    rr = _runner(cfg, ch, fill=0x2222)
    pool_o = oracle.new_pool(cfg, ch.rnd.num_pages, fill=0x2222)
    assert oracle.get().fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents),
                                      pool_o, ch.rnd.num_pages, ch.rnd.block_table) == 0
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    kf = R.to_device_bf16(ch.k_fresh, "cuda")
    kfs = R.to_device_bf16(ch.k_fresh_sel, "cuda")
    vfs = R.to_device_bf16(ch.v_fresh_sel, "cuda")
    rr.alloc_store(int(ch.cost[ch.master]) * cfg.n_layers)
    side = torch.cuda.Stream()
    for _ in range(2):                                   # twice: the second reuses everything
        rr.round_step(kc, vc, kf, kfs, vfs, list(range(cfg.n_agents)), side,
                      torch.cuda.Event(), torch.cuda.Event())
    torch.cuda.synchronize()
    assert int(rr.master_t.item()) == ch.master
    assert np.array_equal(rr.sel_t.cpu().numpy(), ch.sel)
    nnz = ch.store["nnz"]
    assert np.array_equal(rr.store_t["rowptr"].cpu().numpy(), ch.store["rowptr"])
    assert np.array_equal(R.bits_of(rr.store_t["val_k"][:nnz]), ch.store["val_k"])
    assert np.array_equal(R.bits_of(rr.pool_t), pool_o)
    s, bits = rr.get_error()
    assert s == 0 and bits == 0


def test_round_changes_on_a_shared_context_across_streams():
    """Rounds A, B, A through one context, each with its selection, master and encode on a
    side stream overlapped with the re-rotation; B on streams of its own. Nothing synchronizes
    the host between them: the library must order each stream after the round's table
    upload and hold each upload until the work that reads the previous tables is done.
    Every round's outputs are the oracle's, bit for bit."""
    R = _R()
    cfg = synth.qwen7b().replace(n_layers=4, check_layer=2)
    chains = [rk.run_oracle_chain(rk.make_inputs(cfg, seed)) for seed in (501, 502)]
    assert not np.array_equal(chains[0].rnd.perm, chains[1].rnd.perm)
    streams = [(torch.cuda.current_stream(), torch.cuda.Stream()),
               (torch.cuda.Stream(), torch.cuda.Stream())]
    runners, inputs, pools = [], [], []
    ctx = None
    for x, ch in enumerate(chains):
        rr = R.RoundRunner(cfg, ch.rnd.block_len, ch.rnd.hist_len, ch.rnd.perm,
                           ch.rnd.block_table, ch.rnd.num_pages, stream=streams[x][0],
                           pool_fill=0x2222, ctx=ctx)
        ctx = rr.ctx
        rr.alloc_store(int(ch.cost[ch.master]) * cfg.n_layers)
        dev = lambda a: R.to_device_bf16(a, "cuda")
        inputs.append((dev(ch.kc), dev(ch.vc), dev(ch.k_fresh), dev(ch.k_fresh_sel),
                       dev(ch.v_fresh_sel)))
        pool_o = oracle.new_pool(cfg, ch.rnd.num_pages, fill=0x2222)
        assert oracle.get().fused_restore(cfg, ch.desc, ch.master, ch.store,
                                          np.arange(cfg.n_agents), pool_o, ch.rnd.num_pages,
                                          ch.rnd.block_table) == 0
        runners.append(rr)
        pools.append(pool_o)
    torch.cuda.synchronize()
    for x in (0, 1, 0):
        rr = runners[x]
        rr.round_step(*inputs[x], list(range(cfg.n_agents)), streams[x][1], torch.cuda.Event(),
                      torch.cuda.Event())
    torch.cuda.synchronize()
    for rr, ch, pool_o in zip(runners, chains, pools):
        assert int(rr.master_t.item()) == ch.master
        assert np.array_equal(rr.sel_t.cpu().numpy(), ch.sel)
        nnz = ch.store["nnz"]
        assert np.array_equal(rr.store_t["rowptr"].cpu().numpy(), ch.store["rowptr"])
        assert np.array_equal(R.bits_of(rr.store_t["val_k"][:nnz]), ch.store["val_k"])
        assert np.array_equal(R.bits_of(rr.store_t["val_v"][:nnz]), ch.store["val_v"])
        assert np.array_equal(R.bits_of(rr.pool_t), pool_o)
    s, bits = runners[0].get_error()
    assert s == 0 and bits == 0


def test_encode_reads_inputs_written_just_before_it():
    """The encode's main kernel reads the canonical rows before its dependency wait (it is
    scheduled only once the prep kernel has waited for everything earlier). Inputs written
    by a torch kernel on the same stream right before td_diff_encode, with no
    synchronization, must be the ones encoded: the store is the oracle's, bit for bit."""
    R = _R()
    cfg = synth.qwen7b().replace(n_layers=3)
    ch = rk.run_oracle_chain(rk.make_inputs(cfg))
    rr = _runner(cfg, ch)
    sel_t = torch.from_numpy(ch.sel).cuda()
    m = rr.pick_master(sel_t)
    rr.alloc_store(rr.candidate_bound(m))
    kc_true, vc_true = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    kfs, vfs = R.to_device_bf16(ch.k_fresh_sel, "cuda"), R.to_device_bf16(ch.v_fresh_sel, "cuda")
    kc = torch.full_like(kc_true, 7.0)
    vc = torch.full_like(vc_true, -3.0)
    torch.cuda.synchronize()
    with torch.cuda.stream(rr.stream):
        kc.copy_(kc_true)
        vc.copy_(vc_true)
    nnz = rr.diff_encode(kc, vc, kfs, vfs, sel=sel_t)
    torch.cuda.synchronize()
    t = rr.store_t
    assert nnz == ch.store["nnz"]
    assert np.array_equal(R.bits_of(t["master_k"]), ch.store["master_k"])
    assert np.array_equal(R.bits_of(t["master_v"]), ch.store["master_v"])
    assert np.array_equal(t["rowptr"].cpu().numpy(), ch.store["rowptr"])
    assert np.array_equal(R.bits_of(t["val_k"][:nnz]), ch.store["val_k"])
    assert np.array_equal(R.bits_of(t["val_v"][:nnz]), ch.store["val_v"])
    s, bits = rr.get_error()
    assert s == 0 and bits == 0


def test_store_in_host_memory():
    """The store may live in page-locked host memory that the GPU addresses directly
    (NVLink-C2C on GB300): encode writes it there and restore reads it back; both match
    the oracle bit for bit."""
    R = _R()
    cfg = synth.qwen7b().replace(n_layers=3)
    ch = rk.run_oracle_chain(rk.make_inputs(cfg))
    orc = oracle.get()
    pool_o = oracle.new_pool(cfg, ch.rnd.num_pages, fill=0x3333)
    assert orc.fused_restore(cfg, ch.desc, ch.master, ch.store, np.arange(cfg.n_agents), pool_o,
                             ch.rnd.num_pages, ch.rnd.block_table) == 0
    rr = _runner(cfg, ch, fill=0x3333)
    kc, vc = R.to_device_bf16(ch.kc, "cuda"), R.to_device_bf16(ch.vc, "cuda")
    sel_t = torch.from_numpy(ch.sel).cuda()
    m = rr.pick_master(sel_t)
    cap = rr.candidate_bound(m)
    from collective_kv_cache_gb300 import td
    S, E, B, L, N = cfg.n_shared, cfg.elems, cfg.diff_block, cfg.n_layers, cfg.n_agents
    pin = lambda shape, dt: torch.zeros(shape, dtype=dt).pin_memory()
    host = dict(master_k=pin((L, S, E), torch.bfloat16), master_v=pin((L, S, E), torch.bfloat16),
                rowptr=pin((N * L + 1,), torch.int64), block_idx=pin((cap,), torch.int32),
                val_k=pin((cap, B, E), torch.bfloat16), val_v=pin((cap, B, E), torch.bfloat16),
                slot=pin((N * L * rr.nb,), torch.int32))
    rr.store_t = host
    rr.store = td.make_store(host["master_k"], host["master_v"], host["rowptr"],
                             host["block_idx"], host["val_k"], host["val_v"], host["slot"])
    nnz = rr.diff_encode(kc, vc, R.to_device_bf16(ch.k_fresh_sel, "cuda"),
                         R.to_device_bf16(ch.v_fresh_sel, "cuda"), sel=sel_t)
    torch.cuda.synchronize()
    assert nnz == ch.store["nnz"]
    assert np.array_equal(host["rowptr"].numpy(), ch.store["rowptr"])
    assert np.array_equal(host["val_k"][:nnz].view(torch.int16).numpy().view(np.uint16),
                          ch.store["val_k"])
    bits16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits16(host["master_k"]), ch.store["master_k"])
    assert np.array_equal(bits16(host["master_v"]), ch.store["master_v"])
    assert np.array_equal(host["block_idx"][:nnz].numpy(), ch.store["idx"])
    assert np.array_equal(bits16(host["val_v"][:nnz]), ch.store["val_v"])
    from tests.gpu_chain import _check_slots
    _check_slots(host["slot"].numpy(), ch.store, N, L, rr.nb)
    rr.fused_restore(list(range(N)))
    torch.cuda.synchronize()
    assert np.array_equal(R.bits_of(rr.pool_t), pool_o)
    s, bits = rr.get_error()
    assert s == 0 and bits == 0
