"""The library's round formation (segment hashing, KV Collector grouping) against the
oracle, request by request, on the worked example, seeded random prompt sets and the
prompts of the benchmark rounds (host only, no GPU)."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import rounds as OR
from collective_kv_cache_gb300 import synth
from tests.test_rounds_oracle import SEP, _from_round, _random_set, _worked


# ---------------------------------------------------------------- the library
@pytest.fixture(scope="module")
def td():
    from collective_kv_cache_gb300 import build
    build.build()
    from collective_kv_cache_gb300 import td as _td
    return _td


def _fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for byte in data:
        h = ((h ^ byte) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def test_fnv1a_published_vectors():
    # the 64-bit FNV-1a test vectors of its authors' reference suite
    assert _fnv1a64(b"") == 0xCBF29CE484222325
    assert _fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert _fnv1a64(b"foobar") == 0x85944171F73967E8


def test_segment_hash_is_fnv1a_of_the_token_bytes(td):
    rng = np.random.default_rng(3)
    for n in (0, 1, 2, 17, 300):
        t = rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
        assert td.td_segment_hash(t) == _fnv1a64(t.astype("<i4").tobytes())


def _lib_cached(td, cached):
    return None if cached is None else [td.td_segment_hash(np.asarray(b, np.int32)) for b in cached]


def _compare(td, prompts, P, pages=None, cached=None):
    g_o, st_o, n_o = OR.form_rounds(prompts, SEP, P, pages=pages, cached=cached)
    g, st, n = td.td_form_rounds(prompts, SEP, P, pages=pages, cached_hashes=_lib_cached(td, cached))
    assert n == n_o and list(g) == list(g_o) and list(st) == list(st_o)
    for x in range(n):
        mem = [r for r in range(len(prompts)) if g_o[r] == x]
        if st_o[mem[0]] != OR.OK:
            continue
        m_o, bl_o, hl_o, perm_o = OR.group_round(prompts, SEP, g_o, x)
        m, bl, hl, perm = td.td_group_round(prompts, SEP, g, x)
        assert list(m) == list(m_o) and list(bl) == list(bl_o) and list(hl) == list(hl_o)
        assert perm.tolist() == [list(p) for p in perm_o]
    return n


def test_library_worked_example(td):
    prompts, pages, cached, g_exp, st_exp, n_exp, _ = _worked()
    assert _compare(td, prompts, 4, pages=pages, cached=cached) == n_exp
    _compare(td, prompts, 4)


@pytest.mark.parametrize("seed", range(12))
def test_library_matches_oracle_on_random_sets(td, seed):
    prompts, pages, cached, P = _random_set(100 + seed, n_req=120)
    _compare(td, prompts, P, pages=pages, cached=cached)
    _compare(td, prompts, P, pages=None, cached=None)


@pytest.mark.parametrize("name", ["tiny", "qwen7b", "qwen14b", "scale64"])
def test_library_gives_back_the_workload_rounds(td, name):
    cfg = getattr(synth, name)()
    rnd = synth.make_round(cfg)
    prompts, blocks = _from_round(rnd)
    pages = [rnd.block_table[i] for i in range(cfg.n_agents)]
    g, st, n = td.td_form_rounds(prompts, SEP, cfg.page_size, pages=pages,
                                 cached_hashes=_lib_cached(td, blocks))
    assert n == 1 and not st.any()
    mem, bl, hl, perm = td.td_group_round(prompts, SEP, g, 0)
    first = rnd.perm[0]
    assert np.array_equal(bl, rnd.block_len[first]) and np.array_equal(hl, rnd.hist_len)
    assert np.array_equal(first[perm], rnd.perm)


def test_library_edges(td):
    # no requests
    g, st, n = td.td_form_rounds([], SEP, 16)
    assert n == 0 and g.size == 0
    # empty prompts are requests without blocks
    g, st, n = td.td_form_rounds([[], [SEP]], SEP, 16)
    assert list(st) == [OR.NO_BLOCKS, OR.OK] and n == 2
    # a block that is only the separator
    m, bl, hl, perm = td.td_group_round([[SEP]], SEP, [0], 0)
    assert list(bl) == [1] and list(hl) == [0]
    # a group whose members hold different sets is refused
    with pytest.raises(td.TDError):
        td.td_group_round([[SEP, 1], [SEP, 2]], SEP, [0, 0], 0)
    # capacities
    with pytest.raises(td.TDError):
        td.td_group_round([[SEP, 1, SEP, 2]], SEP, [0], 0, cap_blocks=1)
    with pytest.raises(td.TDError):
        td.td_group_round([[SEP, 1], [SEP, 1]], SEP, [0, 0], 0, cap_members=1)
    # a group with no member
    with pytest.raises(td.TDError):
        td.td_group_round([[SEP, 1]], SEP, [0], 3)
    # bad page size
    with pytest.raises(td.TDError):
        td.td_form_rounds([[SEP, 1]], SEP, 0)
