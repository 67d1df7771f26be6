"""Oracle of the round-aware prompt interface and the KV Collector's grouping.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Plain Python over token lists; shared
blocks are matched by their exact token content (no hashing), so the grouping it returns
is the definition the library's hashed version is checked against.

Sources: [R] Summary, Method (1) (reserved separator tokens mark logical block boundaries
so the runtime can hash segments by content and find the blocks agents share) and (2)
(the KV Collector groups requests of a round; incompatible requests fall back to
per-request processing); [R] §2a (segment hashing, grouping); [R] §5 "Batch formation"
(a request joins a group only with the same active prompt length, the same cached span
and disjoint slot mappings); [B] §4.1 (the separator `<TTSEP>`).

READINGS
- A prompt is [private history] [SEP block] [SEP block] ...: the tokens before the first
  separator are the history; every later segment starts at a separator, which belongs to
  it (so block lengths tile the prompt and positions stay contiguous).
- Two blocks are the same block when their tokens are equal.
- A request can join a collective round when it has at least one block, no block twice,
  and every block cached (the caller's set of cached contents). Otherwise it falls back.
- Requests with the same set of blocks (so the same shared span: "same active prompt
  length, same cached span") form one group, in arrival order, as long as none of the
  group's members maps a shared-span position to a page another member also uses
  ("disjoint slot mappings"); a request that would collide opens a new group with the same
  blocks. Groups are numbered in order of their first member.
- A group's round: blocks in the order of its first member's prompt; each member's
  history length and its permutation (slot q holds block perm[q]).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

OK, NO_BLOCKS, REPEATED_BLOCK, NOT_CACHED = 0, 1, 2, 3


def segments(tokens: Sequence[int], sep: int) -> Tuple[int, List[Tuple[int, ...]]]:
    """(history length, list of block contents) of one prompt."""
    tokens = list(tokens)
    cuts = [p for p, tok in enumerate(tokens) if tok == sep]
    hist = cuts[0] if cuts else len(tokens)
    blocks = []
    for q, p in enumerate(cuts):
        end = cuts[q + 1] if q + 1 < len(cuts) else len(tokens)
        blocks.append(tuple(tokens[p:end]))
    return hist, blocks


def form_rounds(prompts: Sequence[Sequence[int]], sep: int, page_size: int,
                pages: Optional[Sequence[Optional[Sequence[int]]]] = None,
                cached: Optional[set] = None):
    """Returns (group_of, status_of, n_groups): group_of[r] is the request's group (every
    fallback request is a group of its own), status_of[r] the fallback reason or OK."""
    n = len(prompts)
    group_of = [-1] * n
    status_of = [OK] * n
    groups: List[dict] = []                  # {"key", "members", "used_pages"}
    for r, toks in enumerate(prompts):
        hist, blocks = segments(toks, sep)
        reason = OK
        if not blocks:
            reason = NO_BLOCKS
        elif len(set(blocks)) != len(blocks):
            reason = REPEATED_BLOCK
        elif cached is not None and any(b not in cached for b in blocks):
            reason = NOT_CACHED
        if reason != OK:
            status_of[r] = reason
            group_of[r] = len(groups)
            groups.append({"key": None, "members": [r], "used_pages": set()})
            continue
        key = frozenset(blocks)
        span = set()
        if pages is not None and pages[r] is not None:
            span_len = sum(len(b) for b in blocks)
            for p in range(hist, hist + span_len):
                span.add(pages[r][p // page_size])
        target = None
        for gi, g in enumerate(groups):
            if g["key"] == key and not (g["used_pages"] & span):
                target = gi
                break
        if target is None:
            target = len(groups)
            groups.append({"key": key, "members": [], "used_pages": set()})
        groups[target]["members"].append(r)
        groups[target]["used_pages"] |= span
        group_of[r] = target
    return group_of, status_of, len(groups)


def group_round(prompts: Sequence[Sequence[int]], sep: int, group_of: Sequence[int], group: int):
    """(members, block_len, hist_len, perm) of one group."""
    members = [r for r, g in enumerate(group_of) if g == group]
    first_hist, first_blocks = segments(prompts[members[0]], sep)
    index: Dict[Tuple[int, ...], int] = {b: j for j, b in enumerate(first_blocks)}
    block_len = [len(b) for b in first_blocks]
    hist_len, perm = [], []
    for r in members:
        hist, blocks = segments(prompts[r], sep)
        hist_len.append(hist)
        perm.append([index[b] for b in blocks])
    return members, block_len, hist_len, perm
