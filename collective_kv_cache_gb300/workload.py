"""Device-side synthetic inputs of a round: canonical K/V and the stand-in for the model's
recompute of the selected tokens (the reused K or canonical V plus the seeded noise of
`synth`). Torch ops on the device, bit for bit the values `synth` gives on the host.

The recompute itself (a model forward) is outside the collective KV path; these tensors
play its output so that the path can be run and timed on synthetic rounds.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import synth


def canonical(cfg: synth.RoundConfig, device, seed: Optional[int] = None, layer_begin=0,
              layer_end=None):
    """Canonical K and V, [nl][S][E] bf16 on the device, layers [layer_begin, layer_end)."""
    layer_end = cfg.n_layers if layer_end is None else layer_end
    nl = layer_end - layer_begin
    kc = torch.empty((nl, cfg.n_shared, cfg.elems), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    for li in range(nl):
        kc[li] = synth.canonical_torch(cfg, "K", layer_begin + li, device, seed)
        vc[li] = synth.canonical_torch(cfg, "V", layer_begin + li, device, seed)
    return kc, vc


def _gather_agent_rows(rr, agent: int, layer_slice, kv: int, pos: np.ndarray):
    P = rr.cfg.page_size
    p = torch.from_numpy(np.asarray(pos, dtype=np.int64)).to(rr.device)
    pages = rr.bt_t[agent].long()[p // P]
    rows = rr.pool_t[layer_slice, kv, pages, p % P]
    return rows.reshape(*rows.shape[:-2], rr.E)


def fresh_check(rr, rnd: synth.Round, seed: Optional[int] = None):
    """Recomputed K at the check layer, [N][S][E] bf16: each agent's reused K plus noise."""
    cfg = rr.cfg
    seed = cfg.seed if seed is None else seed
    pos = rr.positions()
    out = torch.empty((cfg.n_agents, cfg.n_shared, cfg.elems), dtype=torch.bfloat16,
                      device=rr.device)
    tok = torch.arange(cfg.n_shared, dtype=torch.int64, device=rr.device)
    for i in range(cfg.n_agents):
        reused = _gather_agent_rows(rr, i, cfg.check_layer, 0, pos[i])
        pr = torch.from_numpy(rnd.perturbed[i]).to(rr.device)
        noise = synth.noise_rows_torch(seed, "chk", i, cfg.check_layer, tok, pr, cfg.elems)
        out[i] = (reused.float() + noise).to(torch.bfloat16)
    return out


def fresh_selected(rr, rnd: synth.Round, sel: np.ndarray, vc: torch.Tensor,
                   seed: Optional[int] = None, layer_begin=0, layer_end=None,
                   vc_layer0: int = 0):
    """Recomputed K (agent frame) and V at the selected tokens of layers
    [layer_begin, layer_end): two [N][nl][k][E] bf16 tensors. vc holds canonical V of the
    layers from vc_layer0 on."""
    cfg = rr.cfg
    seed = cfg.seed if seed is None else seed
    layer_end = cfg.n_layers if layer_end is None else layer_end
    nl = layer_end - layer_begin
    N, k, E = cfg.n_agents, sel.shape[1], cfg.elems
    kf = torch.empty((N, nl, k, E), dtype=torch.bfloat16, device=rr.device)
    vf = torch.empty_like(kf)
    if k == 0:
        return kf, vf
    pos = rr.positions()
    for i in range(N):
        tok = torch.from_numpy(sel[i].astype(np.int64)).to(rr.device)
        pr = torch.from_numpy(rnd.perturbed[i, sel[i]]).to(rr.device)
        reused = _gather_agent_rows(rr, i, slice(layer_begin, layer_end), 0, pos[i, sel[i]])
        for li in range(nl):
            l = layer_begin + li
            nk = synth.noise_rows_torch(seed, "selK", i, l, tok, pr, E)
            nv = synth.noise_rows_torch(seed, "selV", i, l, tok, pr, E)
            kf[i, li] = (reused[li].float() + nk).to(torch.bfloat16)
            vf[i, li] = (vc[l - vc_layer0, tok].float() + nv).to(torch.bfloat16)
    return kf, vf


def fill_history(rr, rnd: synth.Round, seed: Optional[int] = None):
    """Every agent's private-history K/V (synth.history_torch) written into its pages (the
    round must map its history pages)."""
    cfg = rr.cfg
    P = cfg.page_size
    for i, h in enumerate(rnd.hist_len):
        h = int(h)
        if h == 0:
            continue
        pos = torch.arange(h, dtype=torch.int64, device=rr.device)
        pages = rr.bt_t[i].long()[pos // P]
        if bool((pages < 0).any()):
            raise ValueError("history pages are not mapped")
        for l in range(cfg.n_layers):
            for kv, name in ((0, "K"), (1, "V")):
                rows = synth.history_torch(cfg, i, l, name, h, rr.device, seed)
                rr.pool_t[l, kv, pages, pos % P] = rows.view(h, cfg.n_kv_heads, cfg.head_dim)

