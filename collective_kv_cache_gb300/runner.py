"""Device memory for one All-Gather round and the calls of the collective KV path on it.

PyTorch provides the device allocations and the stream; every stage is one call into the
C-ABI library (collective_kv_cache_gb300.td), whose kernels do all the work.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import td

_BF = torch.bfloat16


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 on the device, same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(_BF)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class RoundRunner:
    """Tensors of one round on one GPU: paged pool, block table, selection, master, store."""

    def __init__(self, cfg, block_len, hist_len, perm, block_table: np.ndarray, num_pages: int,
                 device="cuda", stream: Optional[torch.cuda.Stream] = None,
                 pool_fill: Optional[int] = None, max_agents=None, max_blocks=None,
                 max_shared=None, ctx: Optional["td.Context"] = None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.stream = stream or torch.cuda.current_stream(self.device)
        self.N, self.M = len(hist_len), len(block_len)
        self.S = int(np.sum(block_len))
        self.L, self.E, self.B = cfg.n_layers, cfg.elems, cfg.diff_block
        self.nb = (self.S + self.B - 1) // self.B
        # a context may be shared by several runners (rounds); it must fit each of them
        self.ctx = ctx or td.Context(td.make_shape(cfg), max_agents or self.N,
                                     max_blocks or self.M, max_shared or self.S)
        self.round = td.make_round(block_len, hist_len, perm)
        self._views = None
        self.num_pages = int(num_pages)
        shape = (self.L, 2, self.num_pages, cfg.page_size, cfg.n_kv_heads, cfg.head_dim)
        if pool_fill is None:
            self.pool_t = torch.empty(shape, dtype=_BF, device=self.device)
        else:
            self.pool_t = torch.full(shape, pool_fill, dtype=torch.int16,
                                     device=self.device).view(_BF)
        self.bt_t = torch.from_numpy(np.ascontiguousarray(block_table, dtype=np.int32)).to(self.device)
        self.pool = td.make_paged(self.pool_t, self.bt_t)
        self.master_t = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.cost_t = torch.zeros(self.N, dtype=torch.int64, device=self.device)
        self.dev_t = torch.zeros((self.N, self.S), dtype=torch.float32, device=self.device)
        self.sel_t = None
        self.k = None
        self.store = None
        self.store_t = None

    @property
    def s(self) -> int:
        return self.stream.cuda_stream

    # ------------------------------------------------------------------ stages
    def rerotate(self, kc: torch.Tensor, vc: Optional[torch.Tensor], layer_begin=0,
                 layer_end=None, stream=None):
        """kc, vc hold the layers [layer_begin, layer_end) (row 0 = layer_begin)."""
        layer_end = self.L if layer_end is None else layer_end
        td.td_rerotate_batched(self.ctx.handle, self.round, kc.data_ptr(),
                               vc.data_ptr() if vc is not None else None, layer_begin,
                               layer_end, self.pool, self._s(stream))

    def _s(self, stream) -> int:
        return self.s if stream is None else stream.cuda_stream

    def check_select(self, k_fresh: torch.Tensor, check_layer=None, pct=None, stream=None):
        check_layer = self.cfg.check_layer if check_layer is None else check_layer
        pct = self.cfg.recompute_pct if pct is None else pct
        k = (pct * self.S + 99) // 100
        if self.sel_t is None or self.sel_t.shape[1] != k:
            self.sel_t = torch.zeros((self.N, max(k, 0)), dtype=torch.int32, device=self.device)
        got = td.td_check_select(self.ctx.handle, self.round, check_layer, self.pool,
                                 k_fresh.data_ptr(), pct, self.sel_t.data_ptr() if k else None,
                                 self.dev_t.data_ptr(), self._s(stream))
        assert got == k
        self.k = k
        return self.sel_t

    def pick_master(self, sel: Optional[torch.Tensor] = None, want_host=True, stream=None):
        sel = self.sel_t if sel is None else sel
        k = sel.shape[1]
        return td.td_pick_master(self.ctx.handle, self.round, sel.data_ptr() if k else None, k,
                                 self.cost_t.data_ptr(), self.master_t.data_ptr(),
                                 self._s(stream), want_host=want_host)

    def round_step(self, kc, vc, kf, kfs, vfs, agents, side: torch.cuda.Stream, ev_check,
                   ev_master):
        """One round with the check layer's selection overlapped: the check layer is
        re-rotated first; selection, master choice and the encode (which reads no pages)
        run on `side` while the other layers are re-rotated on the main stream; the restore
        follows on the main stream once both are done. Selection, master and encode use
        their own scratch and re-rotation uses none, so the calls of the two streams may
        overlap; the library orders both streams after the round's table upload."""
        c = self.cfg.check_layer
        main = self.stream
        self.rerotate(kc[c:c + 1], vc[c:c + 1], c, c + 1)
        ev_check.record(main)
        side.wait_event(ev_check)
        self.check_select(kf, stream=side)
        self.pick_master(want_host=False, stream=side)
        self.diff_encode(kc, vc, kfs, vfs, want_nnz=False, stream=side)
        ev_master.record(side)
        if c > 0:
            self.rerotate(kc[:c], vc[:c], 0, c)
        if c + 1 < self.L:
            self.rerotate(kc[c + 1:], vc[c + 1:], c + 1, self.L)
        main.wait_event(ev_master)
        self.fused_restore(agents, frame=0)

    def alloc_store(self, capacity: int, layer_begin=0, layer_end=None):
        layer_end = self.L if layer_end is None else layer_end
        nl = layer_end - layer_begin
        d = self.device
        t = dict(
            master_k=torch.zeros((nl, self.S, self.E), dtype=_BF, device=d),
            master_v=torch.zeros((nl, self.S, self.E), dtype=_BF, device=d),
            rowptr=torch.zeros(self.N * nl + 1, dtype=torch.int64, device=d),
            block_idx=torch.zeros(max(capacity, 1), dtype=torch.int32, device=d),
            val_k=torch.zeros((capacity, self.B, self.E), dtype=_BF, device=d),
            val_v=torch.zeros((capacity, self.B, self.E), dtype=_BF, device=d),
            slot=torch.zeros(self.N * nl * self.nb, dtype=torch.int32, device=d))
        self.store_t = t
        self.store = td.make_store(t["master_k"], t["master_v"], t["rowptr"], t["block_idx"],
                                   t["val_k"], t["val_v"], t["slot"])
        return self.store

    def candidate_bound(self, master: int, layer_begin=0, layer_end=None) -> int:
        layer_end = self.L if layer_end is None else layer_end
        return int(self.cost_t[master].item()) * (layer_end - layer_begin)

    def diff_encode(self, kc, vc, kf, vf, sel=None, master_t=None, layer_begin=0,
                    layer_end=None, want_nnz=True, check=True, stream=None):
        layer_end = self.L if layer_end is None else layer_end
        sel = self.sel_t if sel is None else sel
        master_t = self.master_t if master_t is None else master_t
        k = sel.shape[1]
        return td.td_diff_encode(self.ctx.handle, self.round, master_t.data_ptr(), kc.data_ptr(),
                                 vc.data_ptr(), sel.data_ptr() if k else None, k,
                                 kf.data_ptr() if k else None, vf.data_ptr() if k else None,
                                 layer_begin, layer_end, self.store, self._s(stream),
                                 want_nnz=want_nnz, check=check)

    def fused_restore(self, agents: Sequence[int], layer_begin=None, layer_end=None, frame=0,
                      check=True):
        lb = self.store.layer_begin if layer_begin is None else layer_begin
        le = self.store.layer_end if layer_end is None else layer_end
        return td.td_fused_restore(self.ctx.handle, self.round, self.store, agents, lb, le,
                                   frame, self.pool, self.s, check=check)

    def get_error(self):
        return td.td_get_error(self.ctx.handle, self.s)

    # ------------------------------------------------------------------ comparison baselines
    def agent_views(self):
        """Each agent as a round of its own (its history, its block order, its row of the
        block table) on the same pool: what a per-request system sees."""
        if self._views is None:
            bl, hl, pm = self.round._keep
            pm = pm.reshape(self.N, self.M)
            self._views = []
            for i in range(self.N):
                ctx = td.Context(td.make_shape(self.cfg), 1, self.M, self.S)
                self._views.append((ctx, td.make_round(bl, hl[i:i + 1], pm[i:i + 1]),
                                    td.make_paged(self.pool_t, self.bt_t[i:i + 1])))
        return self._views

    def serial_pic(self, kc, vc, k_fresh):
        """Per-request position-independent caching: for every agent in turn, re-rotate
        the shared blocks into its pages (re-reading the canonical K/V) and run its own
        check-layer selection. Selections land in the rows of sel_t / dev_t."""
        pct, c = self.cfg.recompute_pct, self.cfg.check_layer
        k = (pct * self.S + 99) // 100
        if self.sel_t is None or self.sel_t.shape[1] != k:
            self.sel_t = torch.zeros((self.N, max(k, 0)), dtype=torch.int32, device=self.device)
        for i, (ctx, rnd, pool) in enumerate(self.agent_views()):
            td.td_rerotate_batched(ctx.handle, rnd, kc.data_ptr(), vc.data_ptr(), 0, self.L,
                                   pool, self.s)
            td.td_check_select(ctx.handle, rnd, c, pool, k_fresh[i].data_ptr(), pct,
                               self.sel_t[i].data_ptr() if k else None, self.dev_t[i].data_ptr(),
                               self.s)

    def dense_restore(self, agents: Sequence[int], dense_k: torch.Tensor, dense_v: torch.Tensor):
        """Restore by materialising each agent's dense cache ([L][S][E] K and V), then
        re-rotating it into the agent's pages: the path the fused restore replaces."""
        views = self.agent_views()
        lb, le = self.store.layer_begin, self.store.layer_end
        for a in agents:
            td.td_materialise_mirror(self.ctx.handle, self.round, self.store, a, lb, le,
                                     dense_k.data_ptr(), dense_v.data_ptr(), self.s)
            ctx, rnd, pool = views[a]
            td.td_rerotate_batched(ctx.handle, rnd, dense_k.data_ptr(), dense_v.data_ptr(), lb,
                                   le, pool, self.s)

    # ------------------------------------------------------------------ helpers for inputs
    def positions(self) -> np.ndarray:
        off = td.td_round_offsets(self.round)
        bl = np.asarray(self.round._keep[0], dtype=np.int64)
        start = np.concatenate([[0], np.cumsum(bl)[:-1]])
        tb = np.repeat(np.arange(len(bl)), bl)
        u = np.arange(self.S) - start[tb]
        return off[:, tb] + u[None, :]

    def gather(self, agent: int, layer: int, kv: int, pos: np.ndarray) -> torch.Tensor:
        """Rows of one agent's paged cache at prompt positions -> [n][E] bf16 (device)."""
        P = self.cfg.page_size
        pos_t = torch.from_numpy(np.asarray(pos, dtype=np.int64)).to(self.device)
        pages = self.bt_t[agent].long()[pos_t // P]
        return self.pool_t[layer, kv, pages, pos_t % P].reshape(len(pos), self.E)
