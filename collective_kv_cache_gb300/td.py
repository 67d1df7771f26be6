"""ctypes binding of the C-ABI library (include/td.h): same names, argument marshalling only.

Every stage runs in the library's CUDA kernels; nothing here computes. Importing this
module loads collective_kv_cache_gb300/libtd.so and raises if it has not been built: there
is no fallback path.

Device pointers are passed as Python ints (e.g. torch.Tensor.data_ptr()); streams as the
integer handle of a cudaStream_t (torch.cuda.Stream.cuda_stream). Helpers at the end build
the structs from torch tensors and numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtd.so")

TD_OK = 0
TD_ERR_INVALID_ARG = 1
TD_ERR_CUDA = 2
TD_ERR_CAPACITY = 3
TD_ERR_UNMAPPED_PAGE = 4
TD_ERR_NONFINITE = 5
TD_ERR_DEVICE_TIMEOUT = 6
TD_ERR_SCRATCH_LIMIT = 7


class td_shape(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("page_size", C.c_int32), ("diff_block", C.c_int32), ("rope_theta", C.c_double)]


class td_round(C.Structure):
    _fields_ = [("n_agents", C.c_int32), ("n_blocks", C.c_int32),
                ("block_len", C.POINTER(C.c_int32)), ("hist_len", C.POINTER(C.c_int32)),
                ("perm", C.POINTER(C.c_int32))]


class td_paged(C.Structure):
    _fields_ = [("base", C.c_void_p), ("num_pages", C.c_int64), ("block_table", C.c_void_p),
                ("max_pages_per_agent", C.c_int32)]


class td_diff_store(C.Structure):
    _fields_ = [("master_k", C.c_void_p), ("master_v", C.c_void_p), ("rowptr", C.c_void_p),
                ("block_idx", C.c_void_p), ("val_k", C.c_void_p), ("val_v", C.c_void_p),
                ("slot", C.c_void_p), ("capacity_blocks", C.c_int64),
                ("layer_begin", C.c_int32), ("layer_end", C.c_int32)]


class td_prompt(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("n_tokens", C.c_int64), ("pages", C.c_void_p)]


TD_ROUND_OK, TD_ROUND_NO_BLOCKS, TD_ROUND_REPEATED_BLOCK, TD_ROUND_NOT_CACHED = 0, 1, 2, 3


class TDError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


def _load() -> C.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with collective_kv_cache_gb300.build.build() "
            "(the CUDA library is required; there is no CPU path)")
    lib = C.CDLL(_LIB_PATH)
    P, I32, I64, VP = C.POINTER, C.c_int32, C.c_int64, C.c_void_p
    sig = {
        "td_ctx_create": [P(td_shape), I32, I32, I32, P(VP)],
        "td_ctx_destroy": [VP],
        "td_round_offsets": [P(td_round), VP],
        "td_rerotate_batched": [VP, P(td_round), VP, VP, I32, I32, P(td_paged), VP],
        "td_check_select": [VP, P(td_round), I32, P(td_paged), VP, I32, VP, VP, P(I32), VP],
        "td_pick_master": [VP, P(td_round), VP, I32, VP, VP, P(I32), VP],
        "td_diff_encode": [VP, P(td_round), VP, VP, VP, VP, I32, VP, VP, I32, I32,
                           P(td_diff_store), P(I64), VP],
        "td_fused_restore": [VP, P(td_round), P(td_diff_store), VP, I32, I32, I32, I32,
                             P(td_paged), VP],
        "td_get_error": [VP, VP, P(C.c_uint32)],
        "td_check_select_noalloc": [P(td_shape), P(td_round), I32, P(td_paged), VP, I32, VP,
                                    P(I32), P(C.c_uint32), VP],
        "td_check_select_group": [VP, P(td_round), I32, P(td_paged), VP, I32, VP, VP, VP,
                                  P(I32), VP],
        "td_pick_master_min_deviation": [VP, P(td_round), VP, I32, VP, VP, VP, P(I32), VP],
        "td_materialise_mirror": [VP, P(td_round), P(td_diff_store), I32, I32, I32, VP, VP, VP],
        "td_fused_attention": [VP, P(td_round), P(td_diff_store), P(td_paged), VP, I32, I32, I32,
                               VP, I32, C.c_float, VP, VP, VP],
        "td_paged_attention": [VP, P(td_round), P(td_paged), VP, I32, I32, I32, VP, I32,
                               C.c_float, VP, VP, VP],
        "td_inject_attention_wait_fault": [VP, C.c_uint32],
        "td_form_rounds": [P(td_prompt), I32, I32, I32, VP, I32, VP, VP, P(I32)],
        "td_group_round": [P(td_prompt), I32, I32, VP, I32, I32, I32, VP, P(I32), VP, P(I32),
                           VP, VP],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = C.c_int
    lib.td_segment_hash.argtypes = [VP, I64]
    lib.td_segment_hash.restype = C.c_uint64
    lib.td_status_string.argtypes = [C.c_int]
    lib.td_status_string.restype = C.c_char_p
    return lib


_lib = _load()
EXPORTS = ("td_ctx_create", "td_ctx_destroy", "td_status_string", "td_round_offsets",
           "td_rerotate_batched", "td_check_select", "td_pick_master", "td_diff_encode",
           "td_fused_restore", "td_get_error", "td_check_select_noalloc",
           "td_check_select_group", "td_pick_master_min_deviation", "td_segment_hash",
           "td_form_rounds", "td_group_round", "td_materialise_mirror",
           "td_fused_attention", "td_paged_attention", "td_inject_attention_wait_fault")


def lib_path() -> str:
    return _LIB_PATH


def status_string(s: int) -> str:
    return _lib.td_status_string(int(s)).decode()


def _check(s: int, where: str) -> int:
    if s != TD_OK:
        raise TDError(s, where)
    return s


# ---------------------------------------------------------------- the C calls, same names
def td_ctx_create(shape: td_shape, max_agents: int, max_blocks: int, max_shared: int) -> int:
    out = C.c_void_p()
    _check(_lib.td_ctx_create(C.byref(shape), max_agents, max_blocks, max_shared,
                              C.byref(out)), "td_ctx_create")
    return out.value


def td_ctx_destroy(ctx: int) -> None:
    _check(_lib.td_ctx_destroy(ctx), "td_ctx_destroy")


def td_round_offsets(rnd: td_round) -> np.ndarray:
    off = np.zeros(rnd.n_agents * rnd.n_blocks, dtype=np.int32)
    _check(_lib.td_round_offsets(C.byref(rnd), off.ctypes.data), "td_round_offsets")
    return off.reshape(rnd.n_agents, rnd.n_blocks)


def td_rerotate_batched(ctx, rnd, k_canon, v_canon, layer_begin, layer_end, pool, stream=0,
                        check=True) -> int:
    s = _lib.td_rerotate_batched(ctx, C.byref(rnd), k_canon, v_canon, layer_begin, layer_end,
                                 C.byref(pool), stream)
    return _check(s, "td_rerotate_batched") if check else s


def td_check_select(ctx, rnd, check_layer, pool, k_fresh, recompute_pct, sel, dev_out=None,
                    stream=0, check=True):
    k = C.c_int32(0)
    s = _lib.td_check_select(ctx, C.byref(rnd), check_layer, C.byref(pool), k_fresh,
                             recompute_pct, sel, dev_out, C.byref(k), stream)
    if check:
        _check(s, "td_check_select")
    return (s, k.value) if not check else k.value


def td_pick_master(ctx, rnd, sel, k, cost_out, master_dev, stream=0, want_host=True,
                   check=True):
    m = C.c_int32(-1)
    s = _lib.td_pick_master(ctx, C.byref(rnd), sel, k, cost_out, master_dev,
                            C.byref(m) if want_host else None, stream)
    if check:
        _check(s, "td_pick_master")
        return m.value
    return s, m.value


def td_diff_encode(ctx, rnd, master_dev, k_canon, v_canon, sel, k, k_fresh_sel, v_fresh_sel,
                   layer_begin, layer_end, store: td_diff_store, stream=0, want_nnz=True,
                   check=True):
    nnz = C.c_int64(-1)
    s = _lib.td_diff_encode(ctx, C.byref(rnd), master_dev, k_canon, v_canon, sel, k,
                            k_fresh_sel, v_fresh_sel, layer_begin, layer_end, C.byref(store),
                            C.byref(nnz) if want_nnz else None, stream)
    if check:
        _check(s, "td_diff_encode")
        return nnz.value
    return s, nnz.value


def td_fused_restore(ctx, rnd, store: td_diff_store, agents: Sequence[int], layer_begin,
                     layer_end, frame, pool, stream=0, check=True) -> int:
    ag = np.ascontiguousarray(np.asarray(agents, dtype=np.int32))
    s = _lib.td_fused_restore(ctx, C.byref(rnd), C.byref(store), ag.ctypes.data, len(ag),
                              layer_begin, layer_end, frame, C.byref(pool), stream)
    return _check(s, "td_fused_restore") if check else s


def td_check_select_group(ctx, rnd, check_layer, pool, k_fresh, recompute_pct, sel,
                          dev_out=None, group_dev_out=None, stream=0, check=True):
    k = C.c_int32(0)
    s = _lib.td_check_select_group(ctx, C.byref(rnd), check_layer, C.byref(pool), k_fresh,
                                   recompute_pct, sel, dev_out, group_dev_out, C.byref(k),
                                   stream)
    if check:
        _check(s, "td_check_select_group")
        return k.value
    return s, k.value


def td_pick_master_min_deviation(ctx, rnd, sel, k, dev, score_out, master_dev, stream=0,
                                 want_host=True, check=True):
    m = C.c_int32(-1)
    s = _lib.td_pick_master_min_deviation(ctx, C.byref(rnd), sel, k, dev, score_out,
                                          master_dev, C.byref(m) if want_host else None,
                                          stream)
    if check:
        _check(s, "td_pick_master_min_deviation")
        return m.value
    return s, m.value


def td_fused_attention(ctx, rnd, store, pool, agents, layer_begin, layer_end, q, n_q_heads,
                       scale, out, lse=None, stream=0, check=True) -> int:
    ag = np.ascontiguousarray(agents, dtype=np.int32)
    s = _lib.td_fused_attention(ctx, C.byref(rnd), C.byref(store), C.byref(pool),
                                ag.ctypes.data if ag.size else None, ag.size, layer_begin,
                                layer_end, q, n_q_heads, scale, out, lse, stream)
    return _check(s, "td_fused_attention") if check else s


def td_paged_attention(ctx, rnd, pool, agents, layer_begin, layer_end, q, n_q_heads, scale, out,
                       lse=None, stream=0, check=True) -> int:
    ag = np.ascontiguousarray(agents, dtype=np.int32)
    s = _lib.td_paged_attention(ctx, C.byref(rnd), C.byref(pool),
                                ag.ctypes.data if ag.size else None, ag.size, layer_begin,
                                layer_end, q, n_q_heads, scale, out, lse, stream)
    return _check(s, "td_paged_attention") if check else s


def td_inject_attention_wait_fault(ctx, nbytes: int) -> int:
    return _check(_lib.td_inject_attention_wait_fault(ctx, nbytes),
                  "td_inject_attention_wait_fault")


def td_materialise_mirror(ctx, rnd, store, agent, layer_begin, layer_end, dense_k, dense_v,
                          stream=0) -> int:
    return _check(_lib.td_materialise_mirror(ctx, C.byref(rnd), C.byref(store), agent,
                                             layer_begin, layer_end, dense_k, dense_v, stream),
                  "td_materialise_mirror")


def _prompts(prompts, pages=None):
    keep, arr = [], (td_prompt * max(len(prompts), 1))()
    for r, toks in enumerate(prompts):
        t = np.ascontiguousarray(np.asarray(toks, dtype=np.int32))
        pg = None
        if pages is not None and pages[r] is not None:
            pg = np.ascontiguousarray(np.asarray(pages[r], dtype=np.int32))
            keep.append(pg)
        keep.append(t)
        arr[r] = td_prompt(t.ctypes.data if t.size else None, t.size,
                           pg.ctypes.data if pg is not None else None)
    return arr, keep


def td_segment_hash(tokens) -> int:
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    return int(_lib.td_segment_hash(t.ctypes.data if t.size else None, t.size))


def td_form_rounds(prompts, sep_token, page_size, pages=None, cached_hashes=None):
    """Returns (group_of, status_of, n_groups) as numpy arrays / int."""
    arr, keep = _prompts(prompts, pages)
    n = len(prompts)
    g = np.zeros(max(n, 1), dtype=np.int32)
    st = np.zeros(max(n, 1), dtype=np.int32)
    ng = C.c_int32(0)
    ch = None if cached_hashes is None else np.ascontiguousarray(np.asarray(cached_hashes, dtype=np.uint64))
    _check(_lib.td_form_rounds(arr, n, sep_token, page_size,
                               ch.ctypes.data if ch is not None and ch.size else None,
                               0 if ch is None else ch.size, g.ctypes.data, st.ctypes.data,
                               C.byref(ng)), "td_form_rounds")
    return g[:n].copy(), st[:n].copy(), ng.value


def td_group_round(prompts, sep_token, group_of, group, cap_members=None, cap_blocks=None):
    """Returns (members, block_len, hist_len, perm[n_members][M])."""
    arr, keep = _prompts(prompts)
    n = len(prompts)
    cm = cap_members or max(n, 1)
    cb = cap_blocks or max(max((int(np.count_nonzero(np.asarray(p) == sep_token))
                                for p in prompts), default=1), 1)
    go = np.ascontiguousarray(np.asarray(group_of, dtype=np.int32))
    mem = np.zeros(cm, np.int32)
    bl = np.zeros(cb, np.int32)
    hl = np.zeros(cm, np.int32)
    pm = np.zeros(cm * cb, np.int32)
    nm, nb = C.c_int32(0), C.c_int32(0)
    _check(_lib.td_group_round(arr, n, sep_token, go.ctypes.data, group, cm, cb, mem.ctypes.data,
                               C.byref(nm), bl.ctypes.data, C.byref(nb), hl.ctypes.data,
                               pm.ctypes.data), "td_group_round")
    m, M = nm.value, nb.value
    return mem[:m].copy(), bl[:M].copy(), hl[:m].copy(), pm[:m * M].reshape(m, M).copy()


def td_check_select_noalloc(shape: td_shape, rnd: td_round, check_layer, pool, k_fresh,
                            recompute_pct, sel, stream=0, want_bits=True):
    """Returns (status, k, error bits). Allocates nothing on the device."""
    k = C.c_int32(0)
    bits = C.c_uint32(0)
    s = _lib.td_check_select_noalloc(C.byref(shape), C.byref(rnd), check_layer, C.byref(pool),
                                     k_fresh, recompute_pct, sel, C.byref(k),
                                     C.byref(bits) if want_bits else None, stream)
    return s, k.value, bits.value


def td_get_error(ctx, stream=0):
    bits = C.c_uint32(0)
    s = _lib.td_get_error(ctx, stream, C.byref(bits))
    return s, bits.value


# ---------------------------------------------------------------- marshalling helpers
def make_shape(cfg) -> td_shape:
    return td_shape(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, cfg.page_size, cfg.diff_block,
                    cfg.rope_theta)


def make_round(block_len, hist_len, perm) -> td_round:
    bl = np.ascontiguousarray(block_len, dtype=np.int32)
    hl = np.ascontiguousarray(hist_len, dtype=np.int32)
    pm = np.ascontiguousarray(perm, dtype=np.int32).reshape(-1)
    r = td_round(len(hl), len(bl), bl.ctypes.data_as(C.POINTER(C.c_int32)),
                 hl.ctypes.data_as(C.POINTER(C.c_int32)), pm.ctypes.data_as(C.POINTER(C.c_int32)))
    r._keep = (bl, hl, pm)
    return r


def make_paged(pool_tensor, block_table_tensor) -> td_paged:
    """pool_tensor: torch uint16/bfloat16 [L][2][num_pages][P][H][D] on the GPU;
    block_table_tensor: torch int32 [N][max_lp] on the GPU."""
    p = td_paged(pool_tensor.data_ptr(), pool_tensor.shape[2], block_table_tensor.data_ptr(),
                 block_table_tensor.shape[1])
    p._keep = (pool_tensor, block_table_tensor)
    return p


def make_store(master_k, master_v, rowptr, block_idx, val_k, val_v, slot) -> td_diff_store:
    """torch tensors on the GPU, shaped as td.h describes."""
    cap = val_k.shape[0]
    s = td_diff_store(master_k.data_ptr(), master_v.data_ptr(), rowptr.data_ptr(),
                      block_idx.data_ptr() if cap else None, val_k.data_ptr() if cap else None,
                      val_v.data_ptr() if cap else None, slot.data_ptr(), cap, 0, 0)
    s._keep = (master_k, master_v, rowptr, block_idx, val_k, val_v, slot)
    return s


class Context:
    """Owns a td_ctx handle."""

    def __init__(self, shape: td_shape, max_agents: int, max_blocks: int, max_shared: int):
        self.handle = td_ctx_create(shape, max_agents, max_blocks, max_shared)

    def close(self):
        if self.handle:
            td_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
