"""Parity of the CUDA path with the oracle, bit for bit, on seeded synthetic rounds.

Every stage is compared: the paged pool after re-rotation (including rows that must stay
untouched), the deviations and selections, the master and its costs, the Master's dense
cache, the CSR rows, block indices, diff values and slot map, and the pool after restore
in both frames. Configurations span several tiles, ragged tails (shared spans not a
multiple of 16, blocks that cross diff-block boundaries), page sizes 16, 24 and 32, diff
blocks of 16 and 32 tokens (with a tile that lies wholly in a block's zero tail) and head
layouts of 2x64, 4x128 and 8x128.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from collective_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()


def _mini(**kw):
    base = dict(name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
                block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1,
                recompute_pct=15, perturb_mode="runs", perturb_frac=(0.10, 0.20), seed=77)
    base.update(kw)
    return synth.RoundConfig(**base)


CASES = {
    "tiny": synth.tiny(),
    "mini_ragged_p16": _mini(),
    "mini_ragged_p32": _mini(page_size=32, seed=78),
    "mini_ragged_p24": _mini(page_size=24, seed=79),
    "mini_one_agent": _mini(n_agents=1, seed=80),
    "mini_pct0": _mini(recompute_pct=0, seed=81),
    "mini_pct100": _mini(recompute_pct=100, seed=82),
    "mini_uniform_scatter": _mini(perturb_mode="uniform", seed=83),
    "qwen7b_3layers": synth.qwen7b().replace(n_layers=3),
    "qwen14b_4agents_2layers": synth.qwen14b().replace(n_agents=4, n_layers=2),
    "scale64_2layers": synth.scale64().replace(n_layers=2),
    "density40_p32_8agents_2layers": synth.density(40, page_size=32, pool_bytes=None).replace(
        n_agents=8, n_layers=2),
    # diff block = page size (32 tokens), and 32-token blocks on 16-token pages
    "mini_b32_p32": _mini(diff_block=32, page_size=32, seed=84),
    "mini_b32_p16": _mini(diff_block=32, seed=85),
    "mini_b32_pct100": _mini(diff_block=32, page_size=32, recompute_pct=100, seed=86),
    "mini_b32_pad_tile": _mini(diff_block=32, page_size=32, block_lens=(20, 37, 16, 1), seed=87),
    "mini_b32_uniform_scatter": _mini(diff_block=32, page_size=32, perturb_mode="uniform",
                                      seed=88),
    "qwen7b_b32_p32_3layers": synth.qwen7b().replace(n_layers=3, diff_block=32, page_size=32),
    "density40_b32_p32_8agents_2layers": synth.density(40, page_size=32, pool_bytes=None).replace(
        n_agents=8, n_layers=2, diff_block=32),
    # a shared span beyond one cluster's reach (the selection's many-CTA form), ragged
    "mini_long_span": _mini(n_agents=3, n_layers=2, block_lens=(9000, 6999, 4002), seed=89,
                            hist_range=(0, 300)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_chain_parity(name):
    from tests.gpu_chain import run_and_compare
    run_and_compare(CASES[name])


def test_chain_parity_qwen7b_full():
    """The benchmarked workload at full size: 10 agents, 28 layers, 2560 shared tokens."""
    from tests.gpu_chain import run_and_compare
    run_and_compare(synth.qwen7b(), check_guard=False)
