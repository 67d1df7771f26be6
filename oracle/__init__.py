"""The oracle: a plain, slow CPU definition of the collective KV path (TokenDance).

TEST INFRASTRUCTURE ONLY. The product library never imports, links or runs anything
here; only the test-suite, the smoke check and the benchmark's CPU-baseline leg do.
The C source (td_oracle.c) holds the definitions and their citations; this module
compiles it with gcc and wraps it with ctypes over numpy arrays.

Parity status of each function (what pins it, beyond itself, lives in the tests):
  offsets, rope table, rotate, rerotate     pinned (closed forms, invariants, brute force)
  token deviation, top-k, check-select      pinned (exact sums, brute-force sort)
  pick_master                               pinned (exhaustive set unions)
  pick_master_min_dev, select_group         pinned (exact sums, brute-force sort)
  diff_encode, fused_restore                pinned (bitwise round trip, closed forms)
  compression ratios                        pinned (closed form; the pages' own table)
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "td_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ORC_OK, ORC_ERR_ARG, ORC_ERR_CAPACITY, ORC_ERR_UNMAPPED, ORC_ERR_NONFINITE = 0, 1, 3, 4, 5


def build(force: bool = False, extra_flags: Sequence[str] = (), out: Optional[str] = None) -> str:
    """Compile the oracle (plain C, no contraction of float expressions)."""
    out = out or _LIB
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "td_oracle.h"))):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", *extra_flags, "-o", out + ".tmp", _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


class _Shape(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
                ("page_size", C.c_int), ("diff_block", C.c_int), ("rope_theta", C.c_double)]


class _Round(C.Structure):
    _fields_ = [("n_agents", C.c_int), ("n_blocks", C.c_int),
                ("block_len", C.POINTER(C.c_int32)), ("hist_len", C.POINTER(C.c_int32)),
                ("perm", C.POINTER(C.c_int32))]


class _Pool(C.Structure):
    _fields_ = [("base", C.POINTER(C.c_uint16)), ("num_pages", C.c_int64),
                ("block_table", C.POINTER(C.c_int32)), ("max_lp", C.c_int)]


def _p(a: Optional[np.ndarray], ct):
    if a is None:
        return C.cast(None, C.POINTER(ct))
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ct))


class Oracle:
    """ctypes wrapper; every method takes and returns numpy arrays."""

    def __init__(self, lib_path: Optional[str] = None):
        path = lib_path or build()
        self.lib = C.CDLL(path)
        L = self.lib
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_f32_to_bf16.argtypes = [C.c_float]
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_rope_table.argtypes = [C.c_int64, C.c_int, C.c_double, C.c_void_p, C.c_void_p]
        L.orc_rotate_row.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                     C.c_void_p, C.c_int]
        L.orc_rotate_row_f64.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int64,
                                         C.c_double, C.c_int]
        L.orc_token_dev.restype = C.c_float
        L.orc_token_dev.argtypes = [C.c_void_p, C.c_void_p, C.c_int]
        L.orc_topk.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p]
        L.orc_pick_master.argtypes = [C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p]
        L.orc_pick_master_min_dev.argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_int,
                                              C.c_void_p, C.c_void_p]
        L.orc_select_group.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                       C.c_void_p]
        L.orc_round_ratio.restype = C.c_double
        L.orc_round_ratio.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int64]
        L.orc_mirror_ratio.restype = C.c_double
        L.orc_mirror_ratio.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int64]

    # ---------------------------------------------------------- structs
    @staticmethod
    def shape(cfg) -> _Shape:
        return _Shape(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, cfg.page_size,
                      cfg.diff_block, cfg.rope_theta)

    @staticmethod
    def round_(block_len, hist_len, perm):
        bl = np.ascontiguousarray(block_len, dtype=np.int32)
        hl = np.ascontiguousarray(hist_len, dtype=np.int32)
        pm = np.ascontiguousarray(perm, dtype=np.int32)
        rd = _Round(len(hl), len(bl), _p(bl, C.c_int32), _p(hl, C.c_int32), _p(pm, C.c_int32))
        rd._keep = (bl, hl, pm)
        return rd

    @staticmethod
    def pool(base: np.ndarray, num_pages: int, block_table: np.ndarray):
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        pl = _Pool(_p(base, C.c_uint16), num_pages, _p(bt, C.c_int32), bt.shape[1])
        pl._keep = (base, bt)
        return pl

    # ---------------------------------------------------------- elementary steps
    def f32_to_bf16(self, x: float) -> int:
        return int(self.lib.orc_f32_to_bf16(x))

    def bf16_to_f32(self, h: int) -> float:
        return float(self.lib.orc_bf16_to_f32(h))

    def offsets(self, block_len, hist_len, perm) -> np.ndarray:
        rd = self.round_(block_len, hist_len, perm)
        off = np.zeros((rd.n_agents, rd.n_blocks), dtype=np.int32)
        st = self.lib.orc_offsets(C.byref(rd), _p(off, C.c_int32))
        if st != ORC_OK:
            raise ValueError(f"orc_offsets status {st}")
        return off

    def rope_table(self, a: int, head_dim: int, theta: float):
        c = np.zeros(head_dim // 2, dtype=np.float32)
        s = np.zeros(head_dim // 2, dtype=np.float32)
        self.lib.orc_rope_table(a, head_dim, theta, c.ctypes.data, s.ctypes.data)
        return c, s

    def rotate_row(self, x: np.ndarray, n_heads: int, head_dim: int, a: int, theta: float,
                   inverse: bool = False) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint16)
        c, s = self.rope_table(a, head_dim, theta)
        y = np.zeros_like(x)
        self.lib.orc_rotate_row(x.ctypes.data, y.ctypes.data, n_heads, head_dim, c.ctypes.data,
                                s.ctypes.data, int(inverse))
        return y

    def rotate_row_f64(self, x: np.ndarray, n_heads: int, head_dim: int, a: int, theta: float,
                       inverse: bool = False) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint16)
        y = np.zeros(x.shape, dtype=np.float64)
        self.lib.orc_rotate_row_f64(x.ctypes.data, y.ctypes.data, n_heads, head_dim, a, theta,
                                    int(inverse))
        return y

    def token_dev(self, fresh: np.ndarray, reused: np.ndarray) -> float:
        a = np.ascontiguousarray(fresh, dtype=np.uint16)
        b = np.ascontiguousarray(reused, dtype=np.uint16)
        return float(self.lib.orc_token_dev(a.ctypes.data, b.ctypes.data, a.size))

    def topk(self, dev: np.ndarray, k: int) -> np.ndarray:
        d = np.ascontiguousarray(dev, dtype=np.float32)
        out = np.zeros(k, dtype=np.int32)
        st = self.lib.orc_topk(d.ctypes.data, d.size, k, out.ctypes.data)
        if st != ORC_OK:
            raise FloatingPointError(f"orc_topk status {st}")
        return out

    # ---------------------------------------------------------- the stages
    def rerotate(self, cfg, rnd_desc, k_canon, v_canon, pool_arr, num_pages, block_table,
                 layer_begin=0, layer_end=None) -> int:
        layer_end = cfg.n_layers if layer_end is None else layer_end
        sh = self.shape(cfg)
        rd = self.round_(*rnd_desc)
        pl = self.pool(pool_arr, num_pages, block_table)
        return self.lib.orc_rerotate(C.byref(sh), C.byref(rd), _p(k_canon, C.c_uint16),
                                     _p(v_canon, C.c_uint16), layer_begin, layer_end,
                                     C.byref(pl))

    def check_select(self, cfg, rnd_desc, pool_arr, num_pages, block_table, k_fresh,
                     check_layer=None, pct=None):
        check_layer = cfg.check_layer if check_layer is None else check_layer
        pct = cfg.recompute_pct if pct is None else pct
        sh = self.shape(cfg)
        rd = self.round_(*rnd_desc)
        pl = self.pool(pool_arr, num_pages, block_table)
        N, S = rd.n_agents, int(np.sum(rnd_desc[0]))
        k = (pct * S + 99) // 100
        sel = np.zeros((N, max(k, 0)), dtype=np.int32)
        dev = np.zeros((N, S), dtype=np.float32)
        kout = C.c_int(0)
        st = self.lib.orc_check_select(C.byref(sh), C.byref(rd), check_layer, C.byref(pl),
                                       _p(k_fresh, C.c_uint16), pct, _p(sel, C.c_int32),
                                       _p(dev, C.c_float), C.byref(kout))
        self.last_k = int(kout.value)
        return st, sel, dev

    def pick_master(self, n_shared: int, diff_block: int, sel: np.ndarray):
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        N, k = sel.shape
        cost = np.zeros(N, dtype=np.int64)
        m = self.lib.orc_pick_master(N, n_shared, diff_block, sel.ctypes.data, k, cost.ctypes.data)
        return int(m), cost

    def pick_master_min_dev(self, sel: np.ndarray, dev: np.ndarray):
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        dev = np.ascontiguousarray(dev, dtype=np.float32)
        N, k = sel.shape
        score = np.zeros(N, dtype=np.float64)
        m = self.lib.orc_pick_master_min_dev(N, dev.shape[1], sel.ctypes.data, k, dev.ctypes.data,
                                             score.ctypes.data)
        return int(m), score

    def select_group(self, dev: np.ndarray, k: int):
        dev = np.ascontiguousarray(dev, dtype=np.float32)
        N, S = dev.shape
        row = np.zeros(max(k, 1), dtype=np.int32)
        g = np.zeros(S, dtype=np.float32)
        st = self.lib.orc_select_group(dev.ctypes.data, N, S, k, row.ctypes.data, g.ctypes.data)
        if st != ORC_OK:
            raise FloatingPointError(f"orc_select_group status {st}")
        return row[:k].copy(), g

    def diff_encode(self, cfg, rnd_desc, master, k_canon, v_canon, sel, k_fresh_sel,
                    v_fresh_sel, layer_begin=0, layer_end=None, capacity=None):
        layer_end = cfg.n_layers if layer_end is None else layer_end
        sh = self.shape(cfg)
        rd = self.round_(*rnd_desc)
        N, S, E, B = cfg.n_agents, cfg.n_shared, cfg.elems, cfg.diff_block
        nl = layer_end - layer_begin
        nb = (S + B - 1) // B
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        k = sel.shape[1]
        cap = N * nl * nb if capacity is None else capacity
        mk = np.zeros((nl, S, E), dtype=np.uint16)
        mv = np.zeros((nl, S, E), dtype=np.uint16)
        rowptr = np.zeros(N * nl + 1, dtype=np.int64)
        idx = np.zeros(max(cap, 1), dtype=np.int32)
        vk = np.zeros((max(cap, 1), B, E), dtype=np.uint16)
        vv = np.zeros((max(cap, 1), B, E), dtype=np.uint16)
        nnz = C.c_int64(0)
        st = self.lib.orc_diff_encode(
            C.byref(sh), C.byref(rd), master, _p(k_canon, C.c_uint16), _p(v_canon, C.c_uint16),
            _p(sel, C.c_int32), k, _p(k_fresh_sel, C.c_uint16), _p(v_fresh_sel, C.c_uint16),
            layer_begin, layer_end, _p(mk, C.c_uint16), _p(mv, C.c_uint16),
            _p(rowptr, C.c_int64), _p(idx, C.c_int32), _p(vk, C.c_uint16), _p(vv, C.c_uint16),
            C.c_int64(cap), C.byref(nnz))
        n = int(nnz.value)
        return dict(status=st, nnz=n, master_k=mk, master_v=mv, rowptr=rowptr,
                    idx=idx[:n].copy(), val_k=vk[:n].copy(), val_v=vv[:n].copy())

    def fused_restore(self, cfg, rnd_desc, master, store, agents, pool_arr, num_pages,
                      block_table, layer_begin=0, layer_end=None, frame=0) -> int:
        layer_end = cfg.n_layers if layer_end is None else layer_end
        sh = self.shape(cfg)
        rd = self.round_(*rnd_desc)
        pl = self.pool(pool_arr, num_pages, block_table)
        ag = np.ascontiguousarray(agents, dtype=np.int32)
        vk = store["val_k"] if store["nnz"] else np.zeros((1, cfg.diff_block, cfg.elems), np.uint16)
        vv = store["val_v"] if store["nnz"] else np.zeros((1, cfg.diff_block, cfg.elems), np.uint16)
        ix = store["idx"] if store["nnz"] else np.zeros(1, np.int32)
        return self.lib.orc_fused_restore(
            C.byref(sh), C.byref(rd), master, _p(store["master_k"], C.c_uint16),
            _p(store["master_v"], C.c_uint16), _p(store["rowptr"], C.c_int64),
            _p(np.ascontiguousarray(ix, dtype=np.int32), C.c_int32),
            _p(np.ascontiguousarray(vk), C.c_uint16), _p(np.ascontiguousarray(vv), C.c_uint16),
            _p(ag, C.c_int32), len(ag), layer_begin, layer_end, frame, C.byref(pl))

    def attention(self, cfg, rnd_desc, master, store, agents, pool_arr, num_pages, block_table,
                  q, n_q_heads, scale, layer_begin=0, layer_end=None, from_pool=False):
        """Decode attention from the Master and the diffs (from_pool: every position from
        the pages); q: uint16 bf16 bits [nl][n_list][n_q_heads][D].
        Returns (status, out float64, lse float64)."""
        layer_end = cfg.n_layers if layer_end is None else layer_end
        sh = self.shape(cfg)
        rd = self.round_(*rnd_desc)
        pl = self.pool(pool_arr, num_pages, block_table)
        ag = np.ascontiguousarray(agents, dtype=np.int32)
        nl, D = layer_end - layer_begin, cfg.head_dim
        q = np.ascontiguousarray(q, dtype=np.uint16)
        assert q.shape == (nl, len(ag), n_q_heads, D), q.shape
        out = np.zeros((nl, len(ag), n_q_heads, D), dtype=np.float64)
        lse = np.zeros((nl, len(ag), n_q_heads), dtype=np.float64)
        vk = store["val_k"] if store["nnz"] else np.zeros((1, cfg.diff_block, cfg.elems), np.uint16)
        vv = store["val_v"] if store["nnz"] else np.zeros((1, cfg.diff_block, cfg.elems), np.uint16)
        ix = store["idx"] if store["nnz"] else np.zeros(1, np.int32)
        st = self.lib.orc_attention(
            C.byref(sh), C.byref(rd), master, _p(store["master_k"], C.c_uint16),
            _p(store["master_v"], C.c_uint16), _p(store["rowptr"], C.c_int64),
            _p(np.ascontiguousarray(ix, dtype=np.int32), C.c_int32),
            _p(np.ascontiguousarray(vk), C.c_uint16), _p(np.ascontiguousarray(vv), C.c_uint16),
            C.byref(pl), _p(ag, C.c_int32), len(ag), layer_begin, layer_end,
            _p(q, C.c_uint16), n_q_heads, C.c_double(scale), int(from_pool),
            _p(out, C.c_double), _p(lse, C.c_double))
        return st, out, lse

    def round_ratio(self, cfg, nnz: int) -> float:
        return float(self.lib.orc_round_ratio(cfg.n_agents, cfg.n_layers, cfg.n_shared,
                                              cfg.elems, cfg.diff_block, nnz))

    def mirror_ratio(self, cfg, nnz_mirror: int) -> float:
        return float(self.lib.orc_mirror_ratio(cfg.n_layers, cfg.n_shared, cfg.elems,
                                               cfg.diff_block, nnz_mirror))


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def new_pool(cfg, num_pages: int, fill: int = 0) -> np.ndarray:
    """A host paged pool [L][2][num_pages][P][H][D] of bf16 bits, filled with `fill`."""
    return np.full((cfg.n_layers, 2, num_pages, cfg.page_size, cfg.n_kv_heads, cfg.head_dim),
                   fill, dtype=np.uint16)
