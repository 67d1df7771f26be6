"""Host-side logic of the benchmark: algorithmic byte counts, clock parsing, and the
multi-rank path (independent rounds per rank, max-over-ranks time, summed work) on two
gloo ranks."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

import bench
from collective_kv_cache_gb300 import synth


def test_stage_bytes_closed_form():
    cfg = synth.qwen7b()
    by = bench.stage_bytes(cfg, 10, 28, 384, 22456, 10)
    row = 2560 * 512 * 2
    assert by["rerotate"] == 2 * 28 * row * (1 + 10)
    assert by["select"] == 2 * 10 * 2560 * 512 * 2
    assert by["encode"] == 10 * 28 * 384 * 512 * 4 + 4 * 28 * row + 22456 * (16 * 512 * 4 + 4)
    assert by["restore"] == 2 * 28 * row + 22456 * (16 * 512 * 4 + 4) + 10 * 2 * 28 * row


def test_clock_summary_parses_nvidia_smi_csv():
    cs = bench.ClockSampler("0")
    cs.proc = object()
    cs.out = "\n".join([
        "2026/12/02 06:30:01.100, 0, 1987, 2070, 300.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 06:30:01.150, 0, 2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 06:30:01.200, 0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    s = cs.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_rank_seeds_distinct():
    seeds = {bench.rank_seed(1001, r) for r in range(8)}
    assert len(seeds) == 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank pretends to have timed a different number of milliseconds
        ms = 10.0 + 5.0 * rank
        mx = bench.reduce_max(ms, "cpu")
        work = bench.reduce_sum(100.0 * (rank + 1), "cpu")
        q.put((rank, mx, work, bench.rank_seed(1001, rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_reductions():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [15.0, 15.0]          # max over ranks
    assert [o[2] for o in out] == [300.0, 300.0]        # whole-job work
    assert out[0][3] != out[1][3]                        # independent rounds


def test_threaded_oracle_baseline_matches_single_threaded():
    """The threaded CPU baseline runs the same oracle calls split over layers and agents:
    same selection size and number of diff blocks, and the same restored pool."""
    import bench
    import oracle
    from collective_kv_cache_gb300 import synth
    cfg = synth.tiny().replace(n_layers=4, check_layer=1)
    sub, rnd, kc, vc, orc = bench.oracle_round(cfg, cfg.seed, cfg.n_layers)
    cache = {}
    _, k, nnz = bench.oracle_step(sub, rnd, kc, vc, orc, cache)
    single = cache["restored"]
    _, k_t, nnz_t = bench.oracle_step_threaded(sub, rnd, kc, vc, orc, cache, threads=3)
    cache["executor"].shutdown()
    assert (k_t, nnz_t) == (k, nnz) and nnz > 0
    assert np.array_equal(cache["restored"], single)
    out = bench.cpu_baseline(cfg, cfg.seed, min_seconds=0.0, max_passes=1)
    assert out["threaded"]["value"] > 0 and out["threaded"]["cores"] >= 1


def test_attention_bytes_closed_form():
    cfg = synth.qwen7b()
    hist = [100, 200]
    E, L, S = cfg.elems, cfg.n_layers, cfg.n_shared
    rows = L * 2 * 28
    fused = bench.attention_bytes(cfg, hist, 50, 28, from_pool=False)
    paged = bench.attention_bytes(cfg, hist, 50, 28, from_pool=True)
    assert fused == 300 * L * E * 4 + S * L * E * 4 + 50 * 16 * E * 4 + rows * 128 * 6 + rows * 4
    assert paged == 300 * L * E * 4 + 2 * S * L * E * 4 + rows * 128 * 6 + rows * 4


def test_storage_ratios_match_the_oracle_closed_form():
    """The bench's ratios against the oracle's own closed forms (pinned to the pages'
    storage table by the oracle pins)."""
    import oracle
    cfg = synth.qwen7b()
    orc = oracle.get()
    nnz = 22456
    r = bench.storage_ratios(cfg, nnz, cfg.n_layers)
    assert abs(r["round_ratio"] - orc.round_ratio(cfg, nnz)) < 1e-3
    assert abs(r["per_mirror_ratio"] - orc.mirror_ratio(cfg, nnz // (cfg.n_agents - 1))) < 0.05


def test_diff_density_from_row_pointers():
    cfg = synth.tiny()        # 3 agents, 2 layers, 96 shared tokens -> 6 blocks per layer
    rowptr = np.cumsum([0, 2, 3, 0, 0, 1, 4])        # rows: (a0 l0) (a0 l1) (a1 l0) ...
    d = bench.diff_density(cfg, rowptr, master=1, nl=2)
    assert d["blocks_per_layer"] == 6 and d["max"] == 4
    assert d["mean"] == 2.5 and d["changed_fraction"] == round(2.5 / 6, 4)


def test_round_formation_gives_back_the_round():
    from collective_kv_cache_gb300 import build
    build.build()
    cfg = synth.qwen7b()
    rnd = synth.make_round(cfg)
    r = bench.round_formation(cfg, rnd, reps=1)
    assert r["descriptor_matches_round"]
    assert r["prompt_tokens"] == int(rnd.hist_len.sum()) + cfg.n_agents * cfg.n_shared
