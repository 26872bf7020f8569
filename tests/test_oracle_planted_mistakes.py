"""Mistakes planted in copies of the oracle (on the CPU, never in the CUDA
path) must each be caught by the pins: this is what makes the pins evidence
that the oracle computes what the pages define, not just what it computes.

Each case rewrites one expression of oracle/ds41_oracle.c the way a plausible
slip would (a sign, an offset, a tie rule, a dropped term, a transposed
index), compiles the copy with the oracle's own flags, swaps it in for the
duration of the case, and runs the pins named for it; at least one of them
has to fail.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_out_proj as OP
import test_oracle_pins as PIN

SRC = os.path.join(os.path.dirname(oracle.__file__), "ds41_oracle.c")

# name -> (original text, planted text, pins expected to notice)
CASES = {
    "e2m1 ties to the odd code": (
        "if (d < bestd || (d == bestd && (i % 2 == 0) && (best % 2 == 1))) {",
        "if (d < bestd || (d == bestd && (i % 2 == 1))) {",
        [PIN.test_e2m1_golden_ties, PIN.test_e2m1_sweep_against_midpoints]),
    "e2m1 grid value 3 -> 2.5": (
        "{0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f}",
        "{0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 2.5f, 4.0f, 6.0f}",
        [PIN.test_e2m1_golden_ties, PIN.test_e2m1_sweep_against_midpoints]),
    "e8m0 amax floor dropped": (
        "        if (amax < floor_amax) amax = floor_amax;\n        float s = ds41o_pow2_ceil",
        "        float s = ds41o_pow2_ceil",
        [PIN.test_fp4_quant_golden_examples,
         lambda o: PIN.test_fp4_quant_properties(o, False, 32)]),
    "rotary sign": (
        "x[2 * i] = p00 - p11;", "x[2 * i] = p00 + p11;",
        [PIN.test_rotary_dims_pairs_and_sign, PIN.test_yarn_factor_one_is_plain_rope]),
    "window one position early": (
        "int64_t q = p - win + 1 + j;", "int64_t q = p - win + j;",
        [PIN.test_window_indices_see_exactly_their_window]),
    "latent at the group's last position": (
        "int64_t lpos = crow * ratio;", "int64_t lpos = crow * ratio + ratio - 1;",
        [PIN.test_latent_write_positions_and_rows]),
    "top-k ties to the higher row": (
        "return (x->s < y->s) ? -1 : (x->s > y->s);",
        "return (x->s > y->s) ? -1 : (x->s < y->s);",
        [PIN.test_topk_bruteforce_subsets]),
    "head sum without fma": (
        "acc = fmaf(w[t * Hi + h], r, acc);", "acc = acc + w[t * Hi + h] * r;",
        [PIN.test_indexer_head_sum_is_ordered_fma_chain]),
    "one compressed row visible too few": (
        "int64_t v = (start_pos + t + 1) / ratio;", "int64_t v = (start_pos + t) / ratio;",
        [PIN.test_latent_write_positions_and_rows, PIN.test_topk_bruteforce_subsets,
         lambda o: PIN.test_topk_covering_all_rows_is_dense_causal(o, "decode")]),
    "compress_len counts the unfinished group": (
        "    return (start_pos + m) / ratio;\n}",
        "    return (start_pos + m + ratio - 1) / ratio;\n}",
        [PIN.test_group_counts_by_enumeration,
         lambda o: PIN.test_topk_covering_all_rows_is_dense_causal(o, "chunked")]),
    "new groups counted as m / ratio": (
        "return ds41o_compress_len(m, ratio, start_pos) - start_pos / ratio;",
        "return m / ratio;",
        [PIN.test_group_counts_by_enumeration, PIN.test_latent_write_positions_and_rows]),
    "sink dropped from the denominator": (
        "double den = exp((double)sink[h] - mx);", "double den = 0.0;",
        [PIN.test_one_hot_row_closed_form,
         lambda o: PIN.test_topk_covering_all_rows_is_dense_causal(o, "prefill")]),
    "output side: inverse sign ignored": (
        "ds41o_apply_rotary(x, nh, hd, rd, hp, fc, 1);",
        "ds41o_apply_rotary(x, nh, hd, rd, hp, fc, 0);",
        [OP.test_out_proj_worked_example, OP.test_out_proj_undoes_the_forward_rotation]),
    "output side: positions without start_pos": (
        "hp[h] = start_pos + t;", "hp[h] = t;",
        [OP.test_out_proj_worked_example, OP.test_out_proj_products_against_library_matmul]),
    "output side: wrong group stride of o": (
        "const float* xg = x + g * gw;", "const float* xg = x + g * o_rank;",
        [OP.test_out_proj_groups_are_block_diagonal]),
    "output side: group 0's wo_a rows for every group": (
        "const uint16_t* wr = wo_a + (g * o_rank + r) * gw;",
        "const uint16_t* wr = wo_a + r * gw;",
        [OP.test_out_proj_groups_are_block_diagonal]),
    "output side: og truncated instead of rounded": (
        "gv[g * o_rank + r] = ds41o_f32_to_bf16_rne((float)acc);",
        "{ float fa = (float)acc; uint32_t u; memcpy(&u, &fa, 4); gv[g * o_rank + r] = (uint16_t)(u >> 16); }",
        [OP.test_out_proj_og_rounds_ties_to_even]),
    "output side: wo_b transposed": (
        "acc += (double)ds41o_bf16_to_f32(gv[k]) * (double)ds41o_bf16_to_f32(wr[k]);",
        "acc += (double)ds41o_bf16_to_f32(gv[k]) * (double)ds41o_bf16_to_f32(wo_b[k * dim + j]);",
        [OP.test_out_proj_products_against_library_matmul]),
    "output side: no rotation": (
        "ds41o_apply_rotary(x, nh, hd, rd, hp, fc, 1);", ";",
        [OP.test_out_proj_worked_example]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_planted_mistake_is_caught(orc, name, tmp_path, monkeypatch):
    before, after, pins = CASES[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"{name}: the expression to plant in is gone"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(before, after, 1))
    so = str(tmp_path / "libmut.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so, str(path), "-lm"], check=True)
    lib = ctypes.CDLL(so)
    oracle._sig(lib)
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = 0
    for pin in pins:
        try:
            pin(oracle)
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin noticed: {name}"
