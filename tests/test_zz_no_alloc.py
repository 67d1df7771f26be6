"""td_check_select_noalloc: the selection entry point for callers that may not allocate
device memory. It must give exactly what td_check_select gives (same selection, same k)
on consecutive calls that reuse its fixed scratch, and refuse rounds that do not fit.

Collected last on purpose, so that a run that stops at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from collective_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from collective_kv_cache_gb300 import build
    build.build()
    from collective_kv_cache_gb300 import td
    return td


def _prepared_round(cfg, td):
    """A round re-rotated into its pool by the context path, the synthetic recomputed K at
    the check layer, and the context path's selection."""
    from collective_kv_cache_gb300 import runner as R
    rnd = synth.make_round(cfg)
    kc, vc = synth.canonical_kv(cfg)
    rr = R.RoundRunner(cfg, rnd.block_len, rnd.hist_len, rnd.perm, rnd.block_table,
                       rnd.num_pages)
    rr.rerotate(R.to_device_bf16(kc, "cuda"), R.to_device_bf16(vc, "cuda"))
    pos = rr.positions()
    noise = torch.from_numpy(synth.check_noise(rnd)).cuda()
    kf = torch.stack([(rr.gather(i, cfg.check_layer, 0, pos[i]).float() + noise[i])
                      .to(torch.bfloat16) for i in range(cfg.n_agents)])
    sel_ref = rr.check_select(kf).clone()
    torch.cuda.synchronize()
    return rr, kf, sel_ref


def _mini():
    return synth.RoundConfig(
        name="mini", n_agents=4, n_layers=3, n_kv_heads=2, head_dim=64, page_size=16,
        block_lens=(20, 37, 16, 9), hist_range=(0, 45), check_layer=1, recompute_pct=15,
        seed=77)


def test_noalloc_matches_context_path_on_consecutive_calls(lib):
    td = lib
    rounds = [_prepared_round(_mini(), td),
              _prepared_round(synth.qwen7b().replace(n_layers=3), td)]
    # A, B, A: the second and third calls find the previous call's contents in the scratch
    for idx in (0, 1, 0):
        rr, kf, sel_ref = rounds[idx]
        cfg = rr.cfg
        sel = torch.full_like(sel_ref, -7)
        s, k, bits = td.td_check_select_noalloc(td.make_shape(cfg), rr.round, cfg.check_layer,
                                                rr.pool, kf.data_ptr(), cfg.recompute_pct,
                                                sel.data_ptr(), rr.s)
        assert s == td.TD_OK and bits == 0, (s, bits)
        assert k == sel_ref.shape[1]
        torch.cuda.synchronize()
        assert torch.equal(sel, sel_ref), f"selection differs on round {idx}"


def test_noalloc_rejects_rounds_beyond_its_scratch(lib):
    td = lib
    cfg = synth.RoundConfig(name="big", n_agents=64, n_layers=2, n_kv_heads=1, head_dim=16,
                            page_size=16, block_lens=(20000,), hist_range=(0, 0),
                            hist_fixed=(0,) * 64, check_layer=0)
    rnd = td.make_round(np.array([20000]), np.zeros(64, np.int32), np.zeros((64, 1), np.int32))
    pool_t = torch.zeros((2, 2, 4, 16, 1, 16), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    kf = torch.zeros((16,), dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    s, _, _ = td.td_check_select_noalloc(td.make_shape(cfg), rnd, 0, td.make_paged(pool_t, bt),
                                         kf.data_ptr(), 15, sel.data_ptr())
    assert s == td.TD_ERR_SCRATCH_LIMIT
