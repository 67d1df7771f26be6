"""Pins of the oracle of round-aware prompts and the KV Collector's grouping (host only).

Pins of oracle/rounds.py against facts that do not come from it: a worked example whose
grouping is derived by hand below, prompts built from a known round (history lengths,
block contents, permutations) that must come back out, the separators landing exactly at
the offsets the placement uses, and laws every grouping must obey. Planted mistakes in a
copy of oracle/rounds.py must each fail a pin.
"""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import pytest

import oracle
from oracle import rounds as OR
from collective_kv_cache_gb300 import synth

SEP = 7


# ---------------------------------------------------------------- prompt builders
def _prompt(hist, blocks):
    """[history][SEP block0 tail][SEP block1 tail]...; each block is given WITH its SEP."""
    out = list(hist)
    for b in blocks:
        assert b[0] == SEP
        out += list(b)
    return out


def _block(rng, n, lo=100, hi=50000):
    return (SEP,) + tuple(int(x) for x in rng.integers(lo, hi, size=n - 1))


def _from_round(rnd, seed=5):
    """Prompts of a round: agent i has hist_len[i] private tokens, then block perm[i, q] in
    slot q; blocks have the round's lengths and distinct random contents."""
    rng = np.random.default_rng(seed)
    blocks = [_block(rng, int(L)) for L in rnd.block_len]
    prompts = []
    for i in range(len(rnd.hist_len)):
        hist = [int(x) for x in rng.integers(100, 50000, size=int(rnd.hist_len[i]))]
        prompts.append(_prompt(hist, [blocks[j] for j in rnd.perm[i]]))
    return prompts, blocks


# ---------------------------------------------------------------- the worked example
def _worked():
    """Seven requests, page size 4, every history 4 tokens long (one page).

    b1 = (SEP, 11, 12, 13), b2 = (SEP, 21, 22, 23, 24, 25, 26, 27), b3 = (SEP, 31, 32, 33).
      r0: h  b1 b2      pages [10, 11, 12, 13]   span = positions 4..15 -> pages {11, 12, 13}
      r1: h  b2 b1      pages [10, 21, 22, 23]   same set; span pages {21, 22, 23}: joins r0
                                                   (its history page 10 collides, which does
                                                   not matter: only the span counts)
      r2: h  b1         pages [40, 41]           set {b1}: new group 1
      r3: h  (no SEP)                            NO_BLOCKS: group 2 of its own
      r4: h  b1 b1                               REPEATED_BLOCK: group 3 of its own
      r5: h  b1 b2      pages [50, 12, 51, 52]   set {b1, b2}, but page 12 is r0's: new
                                                   group 4
      r6: h  b2 b1      pages [60, 61, 62, 63]   fits group 0 (the first such) and group 4:
                                                   joins group 0
      r7: h  b3 b1      b3 not cached            NOT_CACHED: group 5 of its own
    """
    b1 = (SEP, 11, 12, 13)
    b2 = (SEP, 21, 22, 23, 24, 25, 26, 27)
    b3 = (SEP, 31, 32, 33)
    h = [1, 2, 3, 4]
    prompts = [_prompt(h, [b1, b2]), _prompt(h, [b2, b1]), _prompt(h, [b1]), list(h) + [5, 6],
               _prompt(h, [b1, b1]), _prompt(h, [b1, b2]), _prompt(h, [b2, b1]),
               _prompt(h, [b3, b1])]
    pages = [[10, 11, 12, 13], [10, 21, 22, 23], [40, 41], [42, 43], [44, 45, 46],
             [50, 12, 51, 52], [60, 61, 62, 63], [70, 71, 72]]
    cached = {b1, b2}
    group_of = [0, 0, 1, 2, 3, 4, 0, 5]
    status_of = [OR.OK, OR.OK, OR.OK, OR.NO_BLOCKS, OR.REPEATED_BLOCK, OR.OK, OR.OK,
                 OR.NOT_CACHED]
    return prompts, pages, cached, group_of, status_of, 6, (b1, b2, b3)


def pin_worked_example(R):
    prompts, pages, cached, g_exp, st_exp, n_exp, (b1, b2, _) = _worked()
    g, st, n = R.form_rounds(prompts, SEP, 4, pages=pages, cached=cached)
    assert list(g) == g_exp and list(st) == st_exp and n == n_exp, (g, st, n)
    # group 0 = r0, r1, r6; blocks in r0's order (b1, b2)
    mem, bl, hl, perm = R.group_round(prompts, SEP, g, 0)
    assert list(mem) == [0, 1, 6]
    assert list(bl) == [len(b1), len(b2)]
    assert list(hl) == [4, 4, 4]
    assert [list(p) for p in perm] == [[0, 1], [1, 0], [1, 0]]
    # without page tables nothing collides: r5 joins group 0 and the later groups shift
    g2, _, n2 = R.form_rounds(prompts, SEP, 4, cached=cached)
    assert list(g2) == [0, 0, 1, 2, 3, 0, 0, 4] and n2 == 5
    # without a cache set every block counts as cached: r7 forms a round of its own
    _, st3, _ = R.form_rounds(prompts, SEP, 4, pages=pages)
    assert st3[7] == OR.OK


def pin_history_pages_do_not_collide(R):
    """Two requests whose histories share a page but whose shared spans do not."""
    b1, b2 = (SEP, 11, 12, 13), (SEP, 21, 22, 23)
    h = [1, 2, 3, 4]
    prompts = [_prompt(h, [b1, b2]), _prompt(h, [b2, b1])]
    g, _, n = R.form_rounds(prompts, SEP, 4, pages=[[10, 11, 12], [10, 21, 22]])
    assert list(g) == [0, 0] and n == 1
    g, _, n = R.form_rounds(prompts, SEP, 4, pages=[[10, 11, 12], [20, 11, 22]])
    assert list(g) == [0, 1] and n == 2


def pin_round_trip_of_a_known_round(R):
    """Prompts built from the 10-agent Qwen-7B round (history lengths, shared blocks in each
    agent's permuted order, Figure 1's layout) give that round back: one group, the blocks
    in agent 0's order, the histories, and each agent's permutation relative to it."""
    for cfg in (synth.tiny(), synth.qwen7b(), synth.scale64().replace(n_agents=12)):
        rnd = synth.make_round(cfg)
        prompts, blocks = _from_round(rnd)
        pages = [rnd.block_table[i] for i in range(cfg.n_agents)]
        g, st, n = R.form_rounds(prompts, SEP, cfg.page_size, pages=pages,
                                 cached=set(blocks))
        assert n == 1 and list(g) == [0] * cfg.n_agents and list(st) == [OR.OK] * cfg.n_agents
        mem, bl, hl, perm = R.group_round(prompts, SEP, g, 0)
        first = list(rnd.perm[0])
        assert list(mem) == list(range(cfg.n_agents))
        assert list(bl) == [int(rnd.block_len[j]) for j in first]
        assert list(hl) == [int(h) for h in rnd.hist_len]
        for i in range(cfg.n_agents):
            assert [first[j] for j in perm[i]] == list(rnd.perm[i])


def pin_separators_sit_at_the_offsets(R):
    """The round the collector derives places block q of agent x exactly where that agent's
    q-th separator stands in its prompt (the placement's offsets, computed by the oracle
    from hist_len, block_len and perm)."""
    cfg = synth.qwen7b()
    rnd = synth.make_round(cfg, seed=11)
    prompts, _ = _from_round(rnd, seed=2)
    g, _, _ = R.form_rounds(prompts, SEP, cfg.page_size)
    _, bl, hl, perm = R.group_round(prompts, SEP, g, 0)
    off = oracle.get().offsets(np.asarray(bl, np.int32), np.asarray(hl, np.int32),
                               np.asarray(perm, np.int32))
    for x, p in enumerate(prompts):
        seps = [t for t, tok in enumerate(p) if tok == SEP]
        for q in range(len(bl)):
            assert off[x, perm[x][q]] == seps[q]


def _random_set(seed, n_req=60, n_blocks=6, page_pool=400, page_size=4):
    """Requests drawing random subsets of a few blocks in random order, some with no block,
    some with a block twice, pages from a small pool so that spans collide."""
    rng = np.random.default_rng(seed)
    blocks = [_block(rng, int(rng.integers(1, 9)), 100, 140) for _ in range(n_blocks)]
    prompts, pages = [], []
    for _ in range(n_req):
        h = [int(x) for x in rng.integers(100, 140, size=int(rng.integers(0, 9)))]
        kind = rng.integers(0, 10)
        if kind == 0:
            chosen = []
        else:
            m = int(rng.integers(1, 3))
            chosen = [blocks[j] for j in rng.choice(n_blocks, size=m, replace=False)]
            if kind == 1:
                chosen = chosen + [chosen[0]]
        p = _prompt(h, chosen)
        prompts.append(p)
        n_pages = (len(p) + page_size - 1) // page_size
        pages.append([int(x) for x in rng.integers(0, page_pool, size=max(n_pages, 1))])
    cached = set(blocks[:-1])
    return prompts, pages, cached, page_size


def pin_grouping_laws(R):
    """On random sets: every group holds one set of blocks; within a group the pages of the
    members' shared spans are pairwise disjoint; group ids follow their first members; a
    request that opened a group collides with every earlier group of its set; fallback
    requests are alone with the right reason."""
    for seed in range(8):
        prompts, pages, cached, P = _random_set(seed)
        g, st, n = R.form_rounds(prompts, SEP, P, pages=pages, cached=cached)
        assert sorted(set(g)) == list(range(n))
        firsts = [list(g).index(x) for x in range(n)]
        assert firsts == sorted(firsts)
        info = []
        for r, p in enumerate(prompts):
            seps = [t for t, tok in enumerate(p) if tok == SEP]
            bl = [tuple(p[a:b]) for a, b in zip(seps, seps[1:] + [len(p)])]
            span = {pages[r][t // P] for t in range(seps[0], len(p))} if seps else set()
            info.append((frozenset(bl), span))
            if not seps:
                assert st[r] == OR.NO_BLOCKS
            elif len(set(bl)) < len(bl):
                assert st[r] == OR.REPEATED_BLOCK
            elif not set(bl) <= cached:
                assert st[r] == OR.NOT_CACHED
            else:
                assert st[r] == OR.OK
            if st[r] != OR.OK:
                assert list(g).count(g[r]) == 1
        for x in range(n):
            mem = [r for r in range(len(prompts)) if g[r] == x]
            if st[mem[0]] != OR.OK:
                continue
            assert len({info[r][0] for r in mem}) == 1
            for a in range(len(mem)):
                for b in range(a + 1, len(mem)):
                    assert not (info[mem[a]][1] & info[mem[b]][1])
            r0 = mem[0]
            for y in range(x):
                earlier = [r for r in range(r0) if g[r] == y]
                if st[earlier[0]] == OR.OK and info[earlier[0]][0] == info[r0][0]:
                    assert any(info[r][1] & info[r0][1] for r in earlier)


PINS = [pin_worked_example, pin_history_pages_do_not_collide, pin_round_trip_of_a_known_round,
        pin_separators_sit_at_the_offsets, pin_grouping_laws]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pins_hold(pin):
    pin(OR)


# ---------------------------------------------------------------- planted mistakes
_SRC = os.path.join(os.path.dirname(OR.__file__), "rounds.py")

MUTANTS = {
    "history_keeps_first_sep": ("hist = cuts[0] if cuts else len(tokens)",
                                "hist = cuts[0] + 1 if cuts else len(tokens)"),
    "sep_ends_a_block": ("blocks.append(tuple(tokens[p:end]))",
                         "blocks.append(tuple(tokens[p + 1:end + 1]))"),
    "ordered_block_key": ("key = frozenset(blocks)", "key = tuple(blocks)"),
    "pages_ignored": ('if g["key"] == key and not (g["used_pages"] & span):',
                      'if g["key"] == key:'),
    "span_from_prompt_start": ("for p in range(hist, hist + span_len):",
                               "for p in range(0, span_len):"),
    "repeats_allowed": ("elif len(set(blocks)) != len(blocks):", "elif False:"),
    "cache_ignored": ("elif cached is not None and any(b not in cached for b in blocks):",
                      "elif False:"),
    "last_fitting_group": ("                target = gi\n                break",
                           "                target = gi"),
    "fallback_shares_an_id": ('groups.append({"key": None, "members": [r], "used_pages": set()})',
                              "pass"),
    "inverse_permutation": ("perm.append([index[b] for b in blocks])",
                            "perm.append(sorted(range(len(blocks)), key=lambda q: index[blocks[q]]))"),
    "history_of_first_member": ("hist_len.append(hist)", "hist_len.append(first_hist)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    path = tmp_path / "rounds_mut.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("rounds_mut", path)
    mut = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mut)
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except Exception as e:  # a failing pin is the expected outcome
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"no pin catches the planted mistake '{name}'"
