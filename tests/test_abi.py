"""The C-ABI library builds, loads and exports every entry point include/td.h declares
(no GPU needed: nothing here launches a kernel)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def td():
    from collective_kv_cache_gb300 import build
    build.build()
    from collective_kv_cache_gb300 import td as _td
    return _td


def _declared():
    text = open(os.path.join(ROOT, "include", "td.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:td_status|const char\*|uint64_t)\s+(td_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(td):
    names = _declared()
    assert len(names) >= 10, names
    lib = ctypes.CDLL(td.lib_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in td.h but not exported"
    assert set(names) == set(td.EXPORTS), set(names) ^ set(td.EXPORTS)


def test_status_strings(td):
    for code in range(8):
        assert td.status_string(code) and td.status_string(code) != "unknown status"


def test_round_offsets_match_oracle(td, orc):
    from collective_kv_cache_gb300 import synth
    for cfg in (synth.tiny(), synth.qwen7b(), synth.scale64()):
        rnd = synth.make_round(cfg)
        got = td.td_round_offsets(td.make_round(rnd.block_len, rnd.hist_len, rnd.perm))
        want = orc.offsets(rnd.block_len, rnd.hist_len, rnd.perm)
        assert np.array_equal(got, want)


def test_round_offsets_rejects_bad_permutation(td):
    r = td.make_round([4, 4], [0, 0], [[0, 0], [1, 0]])
    with pytest.raises(td.TDError) as e:
        td.td_round_offsets(r)
    assert e.value.status == td.TD_ERR_INVALID_ARG
