"""The pins catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake by a textual substitution,
compiles the copy into a temporary library and runs every pin on it: at least one pin
must fail. The oracle itself is never modified.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from tests.test_oracle_pins import PINS

_SRC = os.path.join(os.path.dirname(oracle.__file__), "td_oracle.c")

MUTANTS = {
    # rotation
    "forward_sign": ("y0 = fmaf(x0, c[f], -x1s);", "y0 = fmaf(x0, c[f], x1s);"),
    "inverse_sign": ("y1 = fmaf(x1, c[f], -x0s);", "y1 = fmaf(x1, c[f], x0s);"),
    "interleaved_pairs": ("float x0 = orc_bf16_to_f32(xh[f]);\n      float x1 = orc_bf16_to_f32(xh[f + half]);",
                          "float x0 = orc_bf16_to_f32(xh[2 * f]);\n      float x1 = orc_bf16_to_f32(xh[2 * f + 1]);"),
    "frequency_exponent": ("double inv_freq = pow(theta, -(double)(2 * f) / (double)head_dim);",
                           "double inv_freq = pow(theta, -(double)(f) / (double)head_dim);"),
    "cos_sin_swapped": ("c[f] = (float)cos(ang);\n    s[f] = (float)sin(ang);",
                        "c[f] = (float)sin(ang);\n    s[f] = (float)cos(ang);"),
    # placement
    "offset_after_block": ("off[(int64_t)i * M + j] = (int32_t)pos;\n      pos += rd->block_len[j];",
                           "pos += rd->block_len[j];\n      off[(int64_t)i * M + j] = (int32_t)pos;"),
    "offset_ignores_history": ("int64_t pos = rd->hist_len[i];", "int64_t pos = 0;"),
    "slot_from_wrong_axis": ("* P + pos % P) * E;", "* P + lp % P) * E;"),
    # deviation and selection
    "dev_drops_last_vector": ("for (int v = 0; v < elems / 8; ++v) {", "for (int v = 0; v < elems / 8 - 1; ++v) {"),
    "dev_abs_not_square": ("acc[l] = fmaf(d, d, acc[l]);", "acc[l] = acc[l] + fabsf(d);"),
    "dev_half_tree": ("for (int w = 16; w >= 1; w /= 2)", "for (int w = 8; w >= 1; w /= 2)"),
    "ties_to_higher_token": ("return (a->t > b->t) - (a->t < b->t);", "return (a->t < b->t) - (a->t > b->t);"),
    "smallest_deviation_selected": ("if (a->dev > b->dev) return -1;\n  if (a->dev < b->dev) return 1;",
                                    "if (a->dev < b->dev) return -1;\n  if (a->dev > b->dev) return 1;"),
    "k_rounds_down": ("int k = (recompute_pct * S + 99) / 100;", "int k = (recompute_pct * S) / 100;"),
    # master
    "master_argmax": ("if (best < 0 || c < best_cost)", "if (best < 0 || c > best_cost)"),
    "master_ties_to_higher": ("if (best < 0 || c < best_cost)", "if (best < 0 || c <= best_cost)"),
    "master_counts_intersection": ("c += (mask[(int64_t)i * nb + b] | mask[(int64_t)m * nb + b]) ? 1 : 0;",
                                   "c += (mask[(int64_t)i * nb + b] & mask[(int64_t)m * nb + b]) ? 1 : 0;"),
    "min_dev_argmax": ("if (best < 0 || acc[0] < best_score)", "if (best < 0 || acc[0] > best_score)"),
    "min_dev_drops_last": ("for (int r = 0; r < k; ++r) {\n      int t = sel[(int64_t)i * k + r];\n      if (t < 0 || t >= n_shared) return -ORC_ERR_ARG;",
                           "for (int r = 0; r < k - 1; ++r) {\n      int t = sel[(int64_t)i * k + r];\n      if (t < 0 || t >= n_shared) return -ORC_ERR_ARG;"),
    "group_first_agent_only": ("for (int i = 0; i < n_agents; ++i) s = s + dev[(int64_t)i * n_shared + t];",
                               "for (int i = 0; i < 1; ++i) s = s + dev[(int64_t)i * n_shared + t];"),
    # encode / restore
    "encode_compares_k_only": ("memcmp(xik + (int64_t)t0 * E, xmk + (int64_t)t0 * E, n) != 0 ||\n                        memcmp(xiv + (int64_t)t0 * E, xmv + (int64_t)t0 * E, n) != 0;",
                               "memcmp(xik + (int64_t)t0 * E, xmk + (int64_t)t0 * E, n) != 0;"),
    "encode_no_derotation": ("orc_rotate_row(kf_il + (int64_t)r * E, xk + (int64_t)t * E, H, D, c, s, 1);",
                             "memcpy(xk + (int64_t)t * E, kf_il + (int64_t)r * E, sizeof(uint16_t) * E);"),
    "restore_ignores_diffs": ("int64_t r = row_of_block[t / B];", "int64_t r = -1;"),
    "restore_wrong_direction": ("if (frame == 0) orc_rotate_row(sk, kd, H, D, c, s, 0);",
                                "if (frame == 0) orc_rotate_row(sk, kd, H, D, c, s, 1);"),
    "restore_wrong_row_token": ("val_k + (r * B + t % B) * E", "val_k + (r * B) * E"),
    # attention read from the store
    "attn_drops_history": ("int64_t n = (int64_t)rd->hist_len[a] + S;",
                           "int64_t n = S;"),
    "attn_pool_mode_reads_store": ("int64_t h = from_pool ? n : rd->hist_len[a];",
                                   "int64_t h = rd->hist_len[a];"),
    "attn_ignores_records": ("int64_t r = row_of_block[t / B];\n        const uint16_t* sk = r >= 0 ? val_k + (r * B + t % B) * E : master_k",
                             "int64_t r = -1;\n        const uint16_t* sk = r >= 0 ? val_k + (r * B + t % B) * E : master_k"),
    "attn_rotation_inverse": ("sh->rope_theta, 0);\n        for (int64_t e = 0; e < E; ++e) vx",
                              "sh->rope_theta, 1);\n        for (int64_t e = 0; e < E; ++e) vx"),
    "attn_offset_of_first_block": ("off[(int64_t)a * M + j], sh->rope_theta, 0);",
                                   "off[(int64_t)a * M], sh->rope_theta, 0);"),
    "attn_gqa_modulo": ("int hk = g / G;", "int hk = g % H;"),
    "attn_no_scale": ("sc[p] = scale * d;", "sc[p] = d;"),
    "attn_lse_without_max": ("n > 0 ? mx + log(sum) : -INFINITY;", "n > 0 ? log(sum) : -INFINITY;"),
    "attn_history_from_k_only": ("          double* dst = (kv == 0 ? kx : vx) + p * E;",
                                 "          double* dst = kx + p * E;"),
    # compression
    "ratio_without_master": ("return (double)n_agents * dense / (dense + diff + ptrs);",
                             "return (double)n_agents * dense / (diff + ptrs);"),
    "ratio_values_k_only": ("double diff = (double)nnz * ((double)diff_block * elems * 4.0 + 4.0);",
                            "double diff = (double)nnz * ((double)diff_block * elems * 2.0 + 4.0);"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(_SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_caught(name, src_text, tmp_path):
    old, new = MUTANTS[name]
    assert src_text.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src_text.replace(old, new, 1)
    c_path = tmp_path / "td_oracle.c"
    c_path.write_text(mutated)
    (tmp_path / "td_oracle.h").write_text(open(_SRC.replace(".c", ".h")).read())
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(c_path), "-lm"], check=True, capture_output=True)
    mut = oracle.Oracle(str(so))
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except Exception as e:  # a failing pin is the expected outcome
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"no pin catches the planted mistake '{name}'"
