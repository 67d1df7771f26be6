#!/usr/bin/env python3
"""Benchmark of the collective KV path on GB300: one step = one All-Gather round through
all four stages (re-rotation of the shared blocks into every agent's paged KV, check-layer
deviation and selection, master choice and Master-Mirror encoding, fused restore of every
agent's paged KV), on the Qwen2.5-7B-shaped round: 10 agents, 28 layers, 4 KV heads x 128,
10 shared blocks of 256 tokens, histories uniform on 500..4000 tokens.

Prints one JSON line (rank 0). `value` is the algorithmic HBM bytes of the whole step
divided by its device time, in GB/s; agent-rounds/s and the fraction of the measured HBM
peak ride along. The recompute of the selected tokens (a model forward) is outside the
path: its synthetic stand-in is prepared before timing and stays resident.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own independent round (weak scaling, no collective on
the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
from concurrent.futures import ThreadPoolExecutor
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "restore+reuse KV GB/s (% of GB300 HBM peak); agent-rounds/sec, 7B shape"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (the measured copy peak is the roofline)
LAUNCHES_PER_STEP = 9    # rerotate 1, deviation 1 + top-k 1, master 1, encode 4, restore 1
# DRAM bytes (read + write) per launch of the roofline kernels at the benchmarked size, from
# one ncu capture of these kernels as they are now (dram__bytes_read.sum +
# dram__bytes_write.sum); set an entry to None when its kernel changes.
MEASURED_TRAFFIC = {"qwen7b": {"restore": 2320800000, "rerotate": 1550900000}}
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ------------------------------------------------------------------ shared host logic
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank processes its own independent round."""
    return base_seed + 7919 * rank


def reduce_max(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def stage_bytes(cfg, n_agents: int, nl: int, k: int, nnz: int, n_restored: int) -> dict:
    """Algorithmic HBM bytes of each stage: what the method must move, counted once."""
    S, E, B = cfg.n_shared, cfg.elems, cfg.diff_block
    row = S * E * 2                       # one layer of one tensor, bf16
    rec = B * E * 4 + 4                   # one diff record: K and V values and its index
    return {
        "rerotate": 2 * nl * row + n_agents * 2 * nl * row,
        "select": 2 * n_agents * S * E * 2,
        "master": n_agents * k * 4,
        "encode": n_agents * nl * k * E * 4 + 2 * nl * row + 2 * nl * row + nnz * rec,
        "restore": 2 * nl * row + nnz * rec + n_restored * 2 * nl * row,
    }


def storage_ratios(cfg, nnz: int, nl: int) -> dict:
    """Compression of the round's Master-Mirror store in closed form ([R] §7a: dense KV over
    Master + diffs). One dense agent is nl*S*E bf16 for K and again for V; a diff record
    costs its K and V values plus a 4-byte index; the row pointers 8 bytes each."""
    N, S, E, B = cfg.n_agents, cfg.n_shared, cfg.elems, cfg.diff_block
    dense = nl * S * E * 2 * 2
    rec = B * E * 4 + 4
    store = dense + nnz * rec + 8 * (N * nl + 1)
    per_mirror = dense * (N - 1) / (nnz * rec) if nnz and N > 1 else None
    return {"records": int(nnz), "round_ratio": round(N * dense / store, 3),
            "caches_for_all_agents": round(store / dense, 3),
            "per_mirror_ratio": None if per_mirror is None else round(per_mirror, 3)}


def diff_density(cfg, rowptr, master: int, nl: int) -> dict:
    """Records per (Mirror, layer), from the store's row pointers: how many of a layer's
    diff blocks each Mirror had to keep (the pages' "changed blocks per Mirror")."""
    N = cfg.n_agents
    nb = (cfg.n_shared + cfg.diff_block - 1) // cfg.diff_block
    rp = np.asarray(rowptr, dtype=np.int64)
    per = np.diff(rp).reshape(N, nl)
    mir = np.delete(per, master, axis=0).reshape(-1) if N > 1 else per.reshape(-1)
    if mir.size == 0:
        return None
    q = np.percentile(mir, [10, 50, 90])
    return {"blocks_per_layer": nb, "mean": round(float(mir.mean()), 2),
            "p10": float(q[0]), "p50": float(q[1]), "p90": float(q[2]),
            "max": int(mir.max()), "changed_fraction": round(float(mir.mean()) / nb, 4)}


def round_formation(cfg, rnd, reps: int = 5) -> dict:
    """Host cost of building this round from its agents' token prompts (segment hashing,
    grouping, the round descriptor), and a check that the descriptor is the round's."""
    from collective_kv_cache_gb300 import synth, td
    sep = 151643
    prompts = synth.round_prompts(rnd, sep)
    pages = [rnd.block_table[i] for i in range(cfg.n_agents)]
    t_form = t_group = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        g, st, n = td.td_form_rounds(prompts, sep, cfg.page_size, pages=pages)
        t1 = time.perf_counter()
        members, block_len, hist_len, perm = td.td_group_round(prompts, sep, g, 0)
        t2 = time.perf_counter()
        t_form += t1 - t0
        t_group += t2 - t1
    first = rnd.perm[0]
    same = (n == 1 and not st.any() and np.array_equal(block_len, rnd.block_len[first]) and
            np.array_equal(hist_len, rnd.hist_len) and np.array_equal(first[perm], rnd.perm))
    return {"prompt_tokens": int(sum(len(p) for p in prompts)),
            "form_rounds_ms": round(t_form / reps * 1e3, 3),
            "group_round_ms": round(t_group / reps * 1e3, 3),
            "descriptor_matches_round": bool(same)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""

    def __init__(self, gpu_index: str):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def mark(self, name):
        setattr(self, name, time.time())

    def summary(self):
        """Median SM clock and throttle reasons over the samples taken while our steps ran
        (warm-up and timed steps; the timed region alone is often shorter than the
        sampling period)."""
        if not self.proc:
            return None
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except (ValueError, IndexError):
                continue
        t0 = getattr(self, "load_start", None)
        t1 = getattr(self, "load_end", None)
        under = [r for r in rows if t0 is None or (t0 - 0.05 <= r[0] <= (t1 or 1e18) + 0.05)]
        if not under:
            under = rows
        if not under:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in under:
            for name, val in zip(names, r[3]):
                if val.lower() in ("active", "0x1", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in under),
                "sm_max_mhz": max(r[2] for r in under), "reasons": sorted(reasons),
                "samples": len(under), "window": "warm-up and timed steps"}


# ------------------------------------------------------------------ our arm
def host_store(rr, capacity: int):
    """The round's Master-Mirror store in page-locked host memory that the GPU addresses
    directly (the pages' Storage tier; on GB300 reached over NVLink-C2C)."""
    import torch
    from collective_kv_cache_gb300 import td
    S, E, B, L, N = rr.S, rr.E, rr.B, rr.L, rr.N
    pin = lambda shape, dt: torch.zeros(shape, dtype=dt).pin_memory()
    t = dict(master_k=pin((L, S, E), torch.bfloat16), master_v=pin((L, S, E), torch.bfloat16),
             rowptr=pin((N * L + 1,), torch.int64), block_idx=pin((max(capacity, 1),), torch.int32),
             val_k=pin((capacity, B, E), torch.bfloat16), val_v=pin((capacity, B, E), torch.bfloat16),
             slot=pin((N * L * rr.nb,), torch.int32))
    rr.store_t = t
    rr.store = td.make_store(t["master_k"], t["master_v"], t["rowptr"], t["block_idx"],
                             t["val_k"], t["val_v"], t["slot"])


def setup_round(cfg, seed, device, store_on_host=False):
    """Round inputs resident on the device; the synthetic recompute (reused K plus seeded
    noise) is prepared here, before any timing."""
    import torch
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import synth, workload

    rnd = synth.make_round(cfg, seed)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, device=device)
    kc, vc = workload.canonical(cfg, device, seed)
    rr.rerotate(kc, vc)
    kf = workload.fresh_check(rr, rnd, seed)
    sel = rr.check_select(kf)
    master = rr.pick_master()
    sel_np = sel.cpu().numpy()
    kfs, vfs = workload.fresh_selected(rr, rnd, sel_np, vc, seed)
    bound = rr.candidate_bound(master)
    if store_on_host:
        host_store(rr, max(bound, 1))
    else:
        rr.alloc_store(max(bound, 1))
    nnz = rr.diff_encode(kc, vc, kfs, vfs)
    torch.cuda.synchronize()
    return dict(rr=rr, kc=kc, vc=vc, kf=kf, kfs=kfs, vfs=vfs, k=sel_np.shape[1], nnz=nnz,
                master=master, rnd=rnd)


def workload_config(name: str):
    """qwen7b, qwen14b, scale64, tiny or density<pct>, optionally followed by _p<page size>
    and _b<diff block> (e.g. density40_p32, qwen7b_p32_b32: diff block = page size)."""
    from collective_kv_cache_gb300 import synth
    base, *opts = name.split("_")
    kw = {}
    for o in opts:
        if o[:1] in ("p", "b") and o[1:].isdigit():
            kw["page_size" if o[0] == "p" else "diff_block"] = int(o[1:])
        else:
            raise SystemExit(f"unknown workload {name}")
    if base in synth.CONFIGS:
        cfg = synth.CONFIGS[base]()
    elif base.startswith("density") and base[len("density"):].isdigit():
        cfg = synth.density(int(base[len("density"):]), page_size=kw.pop("page_size", 16))
        opts = [o for o in opts if o[0] != "p"]
    else:
        raise SystemExit(f"unknown workload {name}")
    if kw:
        cfg = cfg.replace(**kw, name=cfg.name + "".join(f"_{o}" for o in opts))
    return cfg


def bench_chunked(args, cfg, seed, device):
    """The same step with encode and restore run in layer chunks (for rounds whose
    recomputed inputs do not fit beside the pool). The synthetic recompute of each chunk
    is built between chunks, untimed; the step time is the sum of the device spans of the
    stages, each measured with CUDA events on the launching stream."""
    import torch
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import synth, workload
    C = args.chunk_layers
    rnd = synth.make_round(cfg, seed)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, device=device)
    kc, vc = workload.canonical(cfg, device, seed)
    rr.rerotate(kc, vc)
    kf = workload.fresh_check(rr, rnd, seed)
    sel = rr.check_select(kf)
    master = rr.pick_master()
    sel_np = sel.cpu().numpy()
    N, L = cfg.n_agents, cfg.n_layers
    agents = list(range(N))
    cost = int(rr.cost_t[master].item())
    stage_ms = {n: 0.0 for n in STAGES}
    nnz_total = 0

    def span(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(rr.stream)
        fn()
        b.record(rr.stream)
        b.synchronize()
        return a.elapsed_time(b)

    for step in range(args.warmup + args.steps):
        timed = step >= args.warmup
        t = {"rerotate": span(lambda: rr.rerotate(kc, vc)),
             "select": span(lambda: rr.check_select(kf)),
             "master": span(lambda: rr.pick_master(want_host=False)),
             "encode": 0.0, "restore": 0.0}
        nnz_step = 0
        for l0 in range(0, L, C):
            l1 = min(L, l0 + C)
            kfs, vfs = workload.fresh_selected(rr, rnd, sel_np, vc, seed, l0, l1)
            if rr.store is None or rr.store.layer_end - rr.store.layer_begin != l1 - l0 \
                    or rr.store_t["val_k"].shape[0] < cost * (l1 - l0):
                rr.store = rr.store_t = None
                torch.cuda.empty_cache()
                rr.alloc_store(max(cost * (l1 - l0), 1), l0, l1)
            rr.store.layer_begin, rr.store.layer_end = l0, l1
            t["encode"] += span(lambda: rr.diff_encode(kc[l0:l1], vc[l0:l1], kfs, vfs,
                                                       layer_begin=l0, layer_end=l1,
                                                       want_nnz=False))
            nnz_step += int(rr.store_t["rowptr"][-1].item())
            t["restore"] += span(lambda: rr.fused_restore(agents))
            del kfs, vfs
        if timed:
            for n in STAGES:
                stage_ms[n] += t[n]
            nnz_total = nnz_step
    s_, bits = rr.get_error()
    if s_ != 0:
        raise RuntimeError(f"device error word {bits:#x}")
    K = args.steps
    stage_ms = {n: v / K for n, v in stage_ms.items()}
    return stage_ms, sel_np.shape[1], nnz_total, master


def run_step(st, agents, events=None):
    rr = st["rr"]
    s = rr.stream
    if events is not None:
        events[0].record(s)
    rr.rerotate(st["kc"], st["vc"])
    if events is not None:
        events[1].record(s)
    rr.check_select(st["kf"])
    if events is not None:
        events[2].record(s)
    rr.pick_master(want_host=False)
    if events is not None:
        events[3].record(s)
    rr.diff_encode(st["kc"], st["vc"], st["kfs"], st["vfs"], want_nnz=False)
    if events is not None:
        events[4].record(s)
    rr.fused_restore(agents, frame=0)
    if events is not None:
        events[5].record(s)


STAGES = ("rerotate", "select", "master", "encode", "restore")


def run_overlapped(st, agents, side, ev_check, ev_master, args):
    """One round with the check layer's selection, the master choice and the encode on a
    second stream, overlapped with the re-rotation of the other layers (--sequential: one
    stream, stages in order)."""
    if args.sequential:
        run_step(st, agents)
        return
    st["rr"].round_step(st["kc"], st["vc"], st["kf"], st["kfs"], st["vfs"], agents, side,
                        ev_check, ev_master)


def bench_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from collective_kv_cache_gb300 import build as _build
    from collective_kv_cache_gb300 import synth

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    cfg = workload_config(args.workload)
    if args.layers:
        cfg = cfg.replace(n_layers=args.layers, name=f"{cfg.name}_first{args.layers}layers")
    seed = rank_seed(cfg.seed, rank)
    if args.chunk_layers is None and args.workload.startswith("density"):
        args.chunk_layers = 8
    if args.chunk_layers:
        return report_chunked(args, cfg, seed, device, rank, world)
    if args.store_on_host:
        cfg = cfg.replace(name=cfg.name + "_store_in_host_memory")
    st = setup_round(cfg, seed, device, store_on_host=args.store_on_host)
    formation = round_formation(cfg, st["rnd"]) if rank == 0 else None
    rr = st["rr"]
    agents = list(range(cfg.n_agents))
    N, L = cfg.n_agents, cfg.n_layers

    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] \
        if world == 1 else str(local_rank)
    clk = ClockSampler(gpu_id if gpu_id.isdigit() else "0").__enter__()
    clk.mark("load_start")
    for _ in range(args.warmup):
        run_step(st, agents)
    torch.cuda.synchronize()
    s, bits = rr.get_error()
    if s != 0:
        raise RuntimeError(f"device error word {bits:#x} after warm-up")

    K = args.steps
    side = torch.cuda.Stream(device, priority=-1)   # the selection's CTAs go first
    ev_c = [torch.cuda.Event() for _ in range(K)]
    ev_m = [torch.cuda.Event() for _ in range(K)]
    for _ in range(2):                      # the overlapped schedule, warmed too
        run_overlapped(st, agents, side, torch.cuda.Event(), torch.cuda.Event(), args)
    graph = None
    if args.graph:
        # one step's launches (both streams) captured once and replayed per step; the
        # round's tables are already on the device, so the calls make no host round trips
        torch.cuda.synchronize()
        main_stream = rr.stream
        rr.stream = torch.cuda.Stream(device)
        graph = torch.cuda.CUDAGraph()
        # thread-local capture: other threads (a process group's watchdog) keep their
        # CUDA calls while this thread captures
        with torch.cuda.graph(graph, stream=rr.stream, capture_error_mode="thread_local"):
            run_overlapped(st, agents, side, torch.cuda.Event(), torch.cuda.Event(), args)
        torch.cuda.synchronize()
        with torch.cuda.stream(rr.stream):
            for _ in range(2):
                graph.replay()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(rr.stream)
    if graph is not None:
        with torch.cuda.stream(rr.stream):
            for i in range(K):
                graph.replay()
    else:
        for i in range(K):
            run_overlapped(st, agents, side, ev_c[i], ev_m[i], args)
    end.record(rr.stream)
    torch.cuda.synchronize()
    if graph is not None:
        rr.stream = main_stream
    clk.mark("load_end")
    clk.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    ms_total = start.elapsed_time(end)
    ms_max = reduce_max(ms_total, device)
    # per-stage attribution: the same steps once more, stages in sequence, one event each
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for i in range(K):
        run_step(st, agents, evs[i])
    torch.cuda.synchronize()
    stage_ms = {name: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) / K
                for j, name in enumerate(STAGES)}
    seq_ms = sum(stage_ms.values())
    s, bits = rr.get_error()
    if s != 0:
        raise RuntimeError(f"device error word {bits:#x} in the timed region")

    comparisons = None if args.no_compare else compare_baselines(st, agents, stage_ms, device)
    attention = None if args.no_attention else bench_attention(cfg, seed, device)
    variants = None if args.no_compare else measure_variants(st, cfg, device)

    by = stage_bytes(cfg, N, L, st["k"], st["nnz"], N)
    step_bytes = sum(by.values())
    total_bytes = reduce_sum(float(step_bytes) * K, device)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    ms_per_step = ms_max / K
    agent_rounds = reduce_sum(float(N) * K, device) / (ms_max * 1e-3)

    # dominant single-kernel stage for the roofline
    dom = max(("rerotate", "restore"), key=lambda n: stage_ms[n])
    achieved = by[dom] / (stage_ms[dom] * 1e-3) / 1e9
    traffic = None if (args.layers or args.store_on_host) else \
        MEASURED_TRAFFIC.get(args.workload, {}).get(dom)

    e2e = bench_e2e(st, agents, cfg, K, device, args) if not args.no_e2e else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, seed, layers=args.cpu_layers)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "agents": N, "layers": L,
                       "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
                       "shared_tokens": cfg.n_shared, "shared_blocks": cfg.n_blocks,
                       "page_size": cfg.page_size, "recompute_pct": cfg.recompute_pct,
                       "history": list(cfg.hist_range), "parallelism": f"independent rounds x{world}",
                       "l2": "inputs larger than L2 (step moves %.2f GB); no flush" % (step_bytes / 1e9)},
            "agent_rounds_per_s": round(agent_rounds, 1),
            "hbm_frac_of_peak": round(value / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
            "hbm_frac_of_nominal": round(value / NOMINAL_HBM_GBS, 4),
            "stages": {n: {"ms": round(stage_ms[n], 5), "bytes": by[n],
                           "gbs": round(by[n] / (stage_ms[n] * 1e-3) / 1e9, 1)} for n in STAGES},
            "diff_blocks": st["nnz"], "selected_per_agent": st["k"], "master": st["master"],
            "round_formation": formation,
            "storage": storage_ratios(cfg, st["nnz"], L),
            "diff_density": diff_density(cfg, rr.store_t["rowptr"].cpu().numpy(), st["master"], L),
            "restore_us_per_agent_layer": round(stage_ms["restore"] * 1e3 / (N * L), 4),
            "host_link": None if not args.store_on_host else {
                "restore_reads_gbs": round((2 * L * cfg.n_shared * cfg.elems * 2 + st["nnz"] *
                                            (cfg.diff_block * cfg.elems * 4 + 4)) / (stage_ms["restore"] * 1e-3) / 1e9, 1),
                "encode_writes_gbs": round((2 * L * cfg.n_shared * cfg.elems * 2 + st["nnz"] *
                                            (cfg.diff_block * cfg.elems * 4 + 4)) / (stage_ms["encode"] * 1e-3) / 1e9, 1)},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "peak_kind": peak_kind},
            "e2e": e2e,
            "gpu_launches": (LAUNCHES_PER_STEP + (0 if args.sequential else
                             (cfg.check_layer > 0) + (cfg.check_layer + 1 < L))) * K,
            "schedule": ("sequential" if args.sequential else
                         "check layer first; selection, master and encode on a second "
                         "stream overlapped with the other layers' re-rotation") +
                        ("; one step captured in a CUDA graph, replayed per step"
                         if args.graph else
                         "; kernels launched from the host, each after the previous with "
                         "programmatic dependent launch"),
            "stages_sequential_ms": round(seq_ms, 5),
            "clocks": clk.summary(),
            "comparisons": comparisons,
            "attention": attention,
            "variants": variants,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def compare_baselines(st, agents, stage_ms, device, reps=3):
    """The pages' two comparisons, run in this process on the same round with the same
    kernels (after the timed region; CUDA events on the launching stream, mean of `reps`):
    serial per-request PIC (one re-rotation and one check-layer selection per agent, each
    re-reading the canonical K/V) against the collective re-rotation + selection, and the
    dense restore (materialise each agent's cache, then re-rotate it into its pages)
    against the fused restore. Both baselines leave bit-identical pages and selections."""
    import torch
    rr = st["rr"]
    dk = torch.empty((rr.L, rr.S, rr.E), dtype=torch.bfloat16, device=device)
    dv = torch.empty_like(dk)
    rr.agent_views()

    def timed(fn):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(rr.stream)
        for _ in range(reps):
            fn()
        b.record(rr.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    serial = timed(lambda: rr.serial_pic(st["kc"], st["vc"], st["kf"]))
    dense = timed(lambda: rr.dense_restore(agents, dk, dv))
    s, bits = rr.get_error()
    if s != 0:
        raise RuntimeError(f"device error word {bits:#x} in the comparison baselines")
    coll = stage_ms["rerotate"] + stage_ms["select"]
    return {"serial_pic_ms": round(serial, 5), "collective_ms": round(coll, 5),
            "collective_speedup": round(serial / coll, 3),
            "dense_restore_ms": round(dense, 5), "fused_restore_ms": round(stage_ms["restore"], 5),
            "fused_speedup": round(dense / stage_ms["restore"], 3),
            "what": "same round and kernels; serial = per-agent re-rotation + selection; "
                    "dense = materialise each agent's cache, then re-rotate it into pages"}


def measure_variants(st, cfg, device, reps=10):
    """The variant readings on the same round, after the timed region: the master with the
    least total deviation of its selected tokens (A6) beside the default union-cost rule,
    and one important set for the whole group (A8) beside the per-agent selection. CUDA
    events on the launching stream, mean of `reps`. The default calls' outputs are put back
    afterwards (the variants write the same selection and master buffers)."""
    import torch
    from collective_kv_cache_gb300 import td
    rr = st["rr"]
    k = rr.sel_t.shape[1]
    sel_keep = rr.sel_t.clone()
    master_keep = rr.master_t.clone()
    score = torch.zeros(cfg.n_agents, dtype=torch.float64, device=device)
    gdev = torch.zeros(cfg.n_shared, dtype=torch.float32, device=device)
    sel_g = torch.zeros_like(rr.sel_t)

    def timed(fn):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(rr.stream)
        for _ in range(reps):
            fn()
        b.record(rr.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    out = {
        "pick_master_ms": timed(lambda: rr.pick_master(want_host=False)),
        "pick_master_min_deviation_ms": timed(lambda: td.td_pick_master_min_deviation(
            rr.ctx.handle, rr.round, rr.sel_t.data_ptr() if k else None, k, rr.dev_t.data_ptr(),
            score.data_ptr(), rr.master_t.data_ptr(), rr.s, want_host=False)),
        "check_select_ms": timed(lambda: rr.check_select(st["kf"])),
        "check_select_group_ms": timed(lambda: td.td_check_select_group(
            rr.ctx.handle, rr.round, cfg.check_layer, rr.pool, st["kf"].data_ptr(),
            cfg.recompute_pct, sel_g.data_ptr() if k else None, rr.dev_t.data_ptr(),
            gdev.data_ptr(), rr.s)),
    }
    rr.check_select(st["kf"])
    rr.sel_t.copy_(sel_keep)
    rr.master_t.copy_(master_keep)
    torch.cuda.synchronize()
    s, bits = rr.get_error()
    if s != 0:
        raise RuntimeError(f"device error word {bits:#x} in the variant readings")
    return {n: round(v, 5) for n, v in out.items()}


def attention_bytes(cfg, hist, nnz, n_q_heads, from_pool: bool) -> int:
    """Algorithmic bytes of one decode-attention call over all layers and agents: each
    agent's history K/V (read from its pages); the shared span's K/V either from the store
    (the Master once for all agents, plus each agent's records, whole blocks) or, over a
    restored cache, from every agent's pages; the bf16 queries, float outputs and lse."""
    L, S, E, B = cfg.n_layers, cfg.n_shared, cfg.elems, cfg.diff_block
    N = len(hist)
    by = int(sum(hist)) * L * E * 4
    by += N * S * L * E * 4 if from_pool else S * L * E * 4 + nnz * B * E * 4
    rows = L * N * n_q_heads
    return by + rows * cfg.head_dim * (2 + 4) + rows * 4


def bench_attention(cfg, seed, device, reps=10):
    """Decode attention of every agent over its context, all layers, read straight from the
    Master and the diffs (td_fused_attention), against the unfused path: restore every
    agent's pages (td_fused_restore), then attend over them (td_paged_attention). Its own
    round with the histories' pages mapped and filled; CUDA events on the launching stream,
    mean of `reps` after warm-up; the working set is far above the L2."""
    import math
    import torch
    from collective_kv_cache_gb300 import runner as R
    from collective_kv_cache_gb300 import synth, td, workload
    nq = cfg.n_q_heads or cfg.n_kv_heads
    rnd = synth.make_round(cfg, seed, map_history=True)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages, device=device)
    kc, vc = workload.canonical(cfg, device, seed)
    rr.rerotate(kc, vc)
    kf = workload.fresh_check(rr, rnd, seed)
    sel = rr.check_select(kf)
    master = rr.pick_master()
    sel_np = sel.cpu().numpy()
    kfs, vfs = workload.fresh_selected(rr, rnd, sel_np, vc, seed)
    rr.alloc_store(max(rr.candidate_bound(master), 1))
    nnz = rr.diff_encode(kc, vc, kfs, vfs)
    del kf, kfs, vfs
    workload.fill_history(rr, rnd, seed)
    N, L = cfg.n_agents, cfg.n_layers
    agents = list(range(N))
    q = R.to_device_bf16(synth.decode_queries(cfg, nq, agents, 0, L, seed), device)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    out_f = torch.empty(q.shape, dtype=torch.float32, device=device)
    out_p = torch.empty_like(out_f)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=device)

    def fused():
        td.td_fused_attention(rr.ctx.handle, rr.round, rr.store, rr.pool, agents, 0, L,
                              q.data_ptr(), nq, scale, out_f.data_ptr(), lse.data_ptr(), rr.s)

    def paged():
        td.td_paged_attention(rr.ctx.handle, rr.round, rr.pool, agents, 0, L, q.data_ptr(), nq,
                              scale, out_p.data_ptr(), lse.data_ptr(), rr.s)

    def restore_then_paged():
        rr.fused_restore(agents)
        paged()

    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(rr.stream)
        for _ in range(reps):
            fn()
        b.record(rr.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    t_fused = timed(fused)
    t_unfused = timed(restore_then_paged)
    t_paged = timed(paged)
    s, bits = rr.get_error()
    if s != 0:
        raise RuntimeError(f"device error word {bits:#x} in the attention comparison")
    diff = float((out_f - out_p).abs().max().item())
    by_f = attention_bytes(cfg, rnd.hist_len, nnz, nq, from_pool=False)
    by_p = attention_bytes(cfg, rnd.hist_len, nnz, nq, from_pool=True)
    by_r = stage_bytes(cfg, N, L, sel_np.shape[1], nnz, N)["restore"]
    peak, peak_kind = measured_peak()
    gbs = by_f / (t_fused * 1e-3) / 1e9
    return {"fused_ms": round(t_fused, 5), "fused_bytes": by_f, "fused_gbs": round(gbs, 1),
            "fused_frac": round(gbs / peak, 4), "peak": peak, "peak_kind": peak_kind,
            "restore_then_paged_ms": round(t_unfused, 5),
            "paged_ms": round(t_paged, 5), "paged_bytes": by_p,
            "paged_gbs": round(by_p / (t_paged * 1e-3) / 1e9, 1),
            "restore_bytes": by_r, "fused_speedup": round(t_unfused / t_fused, 3),
            "query_heads": nq, "max_abs_diff_fused_vs_restored": diff,
            "what": "decode attention of all agents over all layers (history + shared span); "
                    "fused = from the Master and the diffs; unfused = restore all agents' "
                    "pages, then paged attention"}


def report_chunked(args, cfg, seed, device, rank, world):
    local = device.index if device.index is not None else 0
    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0] \
        if world == 1 else str(local)
    clk = ClockSampler(gpu_id if gpu_id.isdigit() else "0").__enter__()
    clk.mark("load_start")
    stage_ms, k, nnz, master = bench_chunked(args, cfg, seed, device)
    clk.mark("load_end")
    clk.__exit__(None, None, None)
    N, L = cfg.n_agents, cfg.n_layers
    ms = sum(stage_ms.values())
    ms_max = reduce_max(ms, device)
    by = stage_bytes(cfg, N, L, k, nnz, N)
    total = reduce_sum(float(sum(by.values())), device)
    value = total / (ms_max * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    dom = max(("rerotate", "restore"), key=lambda n: stage_ms[n])
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "agents": N, "layers": L,
                       "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
                       "shared_tokens": cfg.n_shared, "page_size": cfg.page_size,
                       "recompute_pct": cfg.recompute_pct, "layer_chunk": args.chunk_layers,
                       "timing": "sum of per-stage device spans; the synthetic recompute "
                                 "between layer chunks is not timed",
                       "parallelism": f"independent rounds x{world}"},
            "agent_rounds_per_s": round(reduce_sum(float(N), device) / (ms_max * 1e-3), 1),
            "hbm_frac_of_peak": round(value / peak, 4), "peak_gbs": peak,
            "stages": {n: {"ms": round(stage_ms[n], 5), "bytes": by[n],
                           "gbs": round(by[n] / (stage_ms[n] * 1e-3) / 1e9, 1)} for n in STAGES},
            "diff_blocks": nnz, "selected_per_agent": k, "master": master,
            "roofline": {"bound": "hbm", "kernel": dom,
                         "achieved": round(by[dom] / (stage_ms[dom] * 1e-3) / 1e9, 1),
                         "peak": peak, "unit": "GB/s",
                         "frac": round(by[dom] / (stage_ms[dom] * 1e-3) / 1e9 / peak, 4),
                         "traffic": None, "peak_kind": peak_kind},
            "storage": storage_ratios(cfg, nnz, L),
            "gpu_launches": args.steps * (4 + 5 * ((L + args.chunk_layers - 1) // args.chunk_layers)),
            "clocks": clk.summary(),
            "e2e": None, "cpu_baseline": None,
        }
        print(json.dumps(line), flush=True)


def bench_e2e(st, agents, cfg, K, device, args):
    """Same step through the public calls with HOST inputs: every step's inputs are copied
    from pinned host memory to the device and its result (row pointers, selection, master)
    read back to the host, inside the timed region. The copies run on their own stream into
    two alternating sets of device inputs, so step i + 1's inputs travel while step i
    computes; each copy still waits until the step that last used its set has finished."""
    import torch

    rr = st["rr"]
    names = ("kc", "vc", "kf", "kfs", "vfs")
    host = {n: torch.empty(st[n].shape, dtype=st[n].dtype, pin_memory=True) for n in names}
    for n in names:
        host[n].copy_(st[n])
    sets = [{n: st[n] for n in names}, {n: torch.empty_like(st[n]) for n in names}]
    res = {"rowptr": rr.store_t["rowptr"], "sel": rr.sel_t, "master": rr.master_t}
    res_h = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in res.items()}
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(t.numel() * t.element_size() for t in res.values())
    s = rr.stream
    cs = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device, priority=-1)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        k = i % 2
        cs.wait_event(used[k])
        with torch.cuda.stream(cs):
            for n in names:
                sets[k][n].copy_(host[n], non_blocking=True)
        copied[k].record(cs)

    def compute(i):
        k = i % 2
        s.wait_event(copied[k])
        run_overlapped(dict(st, **sets[k]), agents, side, torch.cuda.Event(), torch.cuda.Event(),
                       args)
        used[k].record(s)
        with torch.cuda.stream(s):
            for n, t in res.items():
                res_h[n].copy_(t, non_blocking=True)

    def steps(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
        s.synchronize()

    steps(3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    cs.wait_event(a)
    steps(K)
    b.record(s)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    by = sum(stage_bytes(cfg, cfg.n_agents, cfg.n_layers, st["k"], st["nnz"],
                         cfg.n_agents).values())
    return {"value": round(by * K / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(ms / K, 4), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "copies": "a copy stream, two alternating input sets: step i+1's inputs travel "
                      "while step i computes"}


# ------------------------------------------------------------------ the oracle on host cores
def oracle_round(cfg, seed, layers):
    """Inputs for the oracle restricted to the first `layers` layers (check layer inside)."""
    import oracle
    from collective_kv_cache_gb300 import synth
    sub = cfg.replace(n_layers=layers)
    rnd = synth.make_round(sub, seed)
    kc, vc = synth.canonical_kv(sub, seed)
    return sub, rnd, kc, vc, oracle.get()


def oracle_step(sub, rnd, kc, vc, orc, cache):
    """One oracle pass over the sample; returns (seconds inside oracle calls, k, nnz).
    The synthetic recompute (reused K plus noise) is built on the first pass and reused;
    it is not timed."""
    import oracle
    from collective_kv_cache_gb300 import synth
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    if "pos" not in cache:
        cache["pos"] = synth.positions(orc.offsets(*desc), rnd.block_len)
    pos = cache["pos"]
    pool = oracle.new_pool(sub, rnd.num_pages)
    t0 = time.perf_counter()
    assert orc.rerotate(sub, desc, kc, vc, pool, rnd.num_pages, rnd.block_table) == 0
    secs = time.perf_counter() - t0
    if "kf" not in cache:
        cache["kf"] = synth.recompute_check(sub, rnd, pos, pool)
    t0 = time.perf_counter()
    st, sel, _ = orc.check_select(sub, desc, pool, rnd.num_pages, rnd.block_table, cache["kf"])
    m, _ = orc.pick_master(sub.n_shared, sub.diff_block, sel)
    secs += time.perf_counter() - t0
    if "kfs" not in cache:
        cache["kfs"], cache["vfs"] = synth.recompute_selected(sub, rnd, pos, pool, vc, sel)
    pool2 = oracle.new_pool(sub, rnd.num_pages)
    t0 = time.perf_counter()
    store = orc.diff_encode(sub, desc, m, kc, vc, sel, cache["kfs"], cache["vfs"])
    orc.fused_restore(sub, desc, m, store, np.arange(sub.n_agents), pool2, rnd.num_pages,
                      rnd.block_table)
    secs += time.perf_counter() - t0
    cache["restored"] = pool2
    return secs, sel.shape[1], store["nnz"]


def oracle_step_threaded(sub, rnd, kc, vc, orc, cache, threads):
    """The same oracle calls partitioned over host threads, with no change to what any
    call computes: re-rotation, encode and restore by layer ranges, the check-layer
    selection by agent (one-agent rounds), the master choice once. ctypes releases the
    interpreter lock inside each call, so the calls run in parallel. Returns (wall
    seconds of the parallel stages, k, nnz); the synthetic recompute comes from `cache`."""
    import oracle
    desc = (rnd.block_len, rnd.hist_len, rnd.perm)
    L, N, bt, npg = sub.n_layers, sub.n_agents, rnd.block_table, rnd.num_pages
    ex = cache.setdefault("executor", ThreadPoolExecutor(threads))
    bounds = np.linspace(0, L, min(threads, L) + 1).round().astype(int)
    chunks = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    if "kfs_chunks" not in cache:
        cache["kfs_chunks"] = {c: (np.ascontiguousarray(cache["kfs"][:, c[0]:c[1]]),
                                   np.ascontiguousarray(cache["vfs"][:, c[0]:c[1]]))
                               for c in chunks}
        cache["kf_rows"] = [np.ascontiguousarray(cache["kf"][i:i + 1]) for i in range(N)]
    pool = oracle.new_pool(sub, npg)
    pool2 = oracle.new_pool(sub, npg)
    t0 = time.perf_counter()
    assert all(st == 0 for st in ex.map(
        lambda c: orc.rerotate(sub, desc, kc, vc, pool, npg, bt, c[0], c[1]), chunks))

    def one_agent(i):
        d = (rnd.block_len, rnd.hist_len[i:i + 1], rnd.perm[i:i + 1])
        st, sel_i, _ = orc.check_select(sub, d, pool, npg, bt[i:i + 1], cache["kf_rows"][i])
        assert st == 0
        return sel_i[0]

    sel = np.stack(list(ex.map(one_agent, range(N))))
    m, _ = orc.pick_master(sub.n_shared, sub.diff_block, sel)

    def encode_restore(c):
        kfs, vfs = cache["kfs_chunks"][c]
        store = orc.diff_encode(sub, desc, m, kc, vc, sel, kfs, vfs, c[0], c[1])
        assert store["status"] == 0
        assert orc.fused_restore(sub, desc, m, store, np.arange(N), pool2, npg, bt, c[0],
                                 c[1]) == 0
        return store["nnz"]

    nnz = sum(ex.map(encode_restore, chunks))
    secs = time.perf_counter() - t0
    cache["restored"] = pool2
    return secs, sel.shape[1], nnz


def cpu_baseline(cfg, seed, layers=None, min_seconds=10.0, max_passes=8):
    """The oracle, single-threaded, on the same round (all layers unless `layers`),
    repeated until at least `min_seconds` of oracle time have accumulated."""
    layers = cfg.n_layers if layers is None else layers
    sub, rnd, kc, vc, orc = oracle_round(cfg, seed, layers)
    cache = {}
    secs, passes, k, nnz = 0.0, 0, 0, 0
    while passes < max_passes and (passes == 0 or secs < min_seconds):
        t, k, nnz = oracle_step(sub, rnd, kc, vc, orc, cache)
        secs += t
        passes += 1
    by = sum(stage_bytes(sub, sub.n_agents, layers, k, nnz, sub.n_agents).values()) * passes
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    tsecs, tpasses = 0.0, 0
    while tpasses < max_passes and (tpasses == 0 or tsecs < min_seconds / 2):
        t, k_t, nnz_t = oracle_step_threaded(sub, rnd, kc, vc, orc, cache, threads)
        assert (k_t, nnz_t) == (k, nnz)
        tsecs += t
        tpasses += 1
    cache["executor"].shutdown()
    tby = by / passes * tpasses
    return {"value": round(by / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "seconds": round(secs, 2),
            "threaded": {"value": round(tby / tsecs / 1e9, 4), "cores": threads,
                         "seconds": round(tsecs, 2), "passes": tpasses,
                         "how": "the same oracle calls split over threads: re-rotation, "
                                "encode and restore by layer ranges, selection by agent"},
            "sample": f"{passes} single-threaded passes of the plain C oracle over the same "
                      f"round, layers 0..{layers - 1} of {cfg.n_layers} (all {cfg.n_agents} "
                      f"agents, all {cfg.n_shared} shared tokens)"}


def bench_reference(args, rank, world):
    """The reference arm: the oracle as it stands, on the host cores, same metric."""
    if rank != 0:
        return
    from collective_kv_cache_gb300 import synth
    cfg = synth.CONFIGS[args.workload]()
    layers = args.ref_layers
    sub, rnd, kc, vc, orc = oracle_round(cfg, cfg.seed, layers)
    cache = {}
    for _ in range(args.warmup):
        oracle_step(sub, rnd, kc, vc, orc, cache)
    tot, k, nnz = 0.0, 0, 0
    for _ in range(args.steps):
        secs, k, nnz = oracle_step(sub, rnd, kc, vc, orc, cache)
        tot += secs
    by = sum(stage_bytes(sub, sub.n_agents, layers, k, nnz, sub.n_agents).values())
    value = by * args.steps / tot / 1e9
    sample = (f"each step: the round restricted to layers 0..{layers - 1} of {cfg.n_layers}, "
              f"all agents and tokens, single-threaded plain C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "agents": cfg.n_agents, "layers": cfg.n_layers,
                   "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
                   "shared_tokens": cfg.n_shared, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen7b")
    ap.add_argument("--chunk-layers", type=int, default=None,
                    help="run encode and restore in layer chunks (density workloads: 8)")
    ap.add_argument("--layers", type=int, default=None,
                    help="same shape with fewer layers (small profiling case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--store-on-host", action="store_true",
                    help="keep the Master-Mirror store in page-locked host memory (encode "
                         "writes it, restore reads it, over the host link)")
    ap.add_argument("--sequential", action="store_true",
                    help="one stream, stages in order (no overlap of the selection)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the serial-PIC and dense-restore comparison baselines")
    ap.add_argument("--no-attention", action="store_true",
                    help="skip the fused-attention measurement")
    ap.add_argument("--graph", action="store_true",
                    help="replay one captured CUDA graph per step instead of launching every "
                         "step's kernels from the host")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch from the host (the default; kept for older command lines)")
    ap.add_argument("--cpu-layers", type=int, default=None)
    ap.add_argument("--ref-layers", type=int, default=4)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        bench_reference(args, rank, world)
    else:
        bench_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
