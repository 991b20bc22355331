"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle.c, plants one plausible mistake (a wrong index, a
dropped term, a wrong sign, a transposed operand, a wrong rounding or
threshold rule), builds it with the oracle's own flags, and runs the pin
battery of test_oracle_pins.py against that build in a child process (a
planted mistake may also crash).  The unmodified source must pass the same
battery, so the harness itself is checked too.  Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "getblock_index": ("return ufr[(W + p - 1 - s) % W];", "return ufr[(W + p - s) % W];"),
    "drop_own_input_last_step": ("float v = ring_func(op, this_buffer[k], x);",
                                 "float v = this_buffer[k];"),
    "sum_sign": ("return acc + x; /* sum and avg */", "return acc - x; /* sum and avg */"),
    "max_operand": ("if (acc > x) return acc;", "if (acc > x) return x;"),
    "max_signed_zero": ("(signbit(acc) && signbit(x))", "(signbit(acc) || signbit(x))"),
    "segment_offset": ("*off = (int64_t)j * q + (j < r ? j : r);", "*off = (int64_t)j * q;"),
    "bf16_round_half_up": ("u += 0x7FFFu + lsb;", "u += 0x8000u;"),
    "bf16_widen_shift": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    "avg_scale_dropped": ("if (op == ORACLE_AVG) v = v * scale;", ";"),
    "avg_divides_by_w": ("if (op == ORACLE_AVG) v = v * scale;",
                         "if (op == ORACLE_AVG) v = v / (float)W;"),
    "avg_casts_before_scale": ("if (op == ORACLE_AVG) v = v * scale;",
                               "if (op == ORACLE_AVG) v = round_to(v, dtype) * scale;"),
    "fusion_threshold_strict": ("size + counts[t] * es <= threshold_bytes",
                                "size + counts[t] * es < threshold_bytes"),
    "allgather_block": ("int b = ufr[(p - s + W) % W];", "int b = ufr[(p + s) % W];"),
    "ring_position_vs_user_rank": ("float x = load_elem(in[me], boff + k, dtype);",
                                   "float x = load_elem(in[p], boff + k, dtype);"),
    "buffer_to_self": ("float* next_buffer = nxt + (int64_t)((p + 1) % W) * maxlen;",
                       "float* next_buffer = nxt + (int64_t)p * maxlen;"),
    "pack_offset": ("memcpy((char*)fused[u] + offset * es, tensors[(int64_t)u * T + t],",
                    "memcpy((char*)fused[u], tensors[(int64_t)u * T + t],"),
    "last_step_early": ("} else if (s < W - 1) {", "} else if (s < W - 2) {"),
    "min_operand": ("if (acc < x) return acc;", "if (acc < x) return x;"),
    "min_signed_zero": ("(signbit(acc) || signbit(x)) ? -0.0f", "(signbit(acc) && signbit(x)) ? -0.0f"),
    "prod_is_sum": ("if (op == ORACLE_PROD) return acc * x;", "if (op == ORACLE_PROD) return acc + x;"),
    "f16_round_half_up": ("if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) ++r;",
                          "if (rem >= 0x1000u) ++r;"),
    "f16_subnormal_shift": ("const int shift = 14 - e; /* 14..24 */",
                            "const int shift = 13 - e; /* 14..24 */"),
    "hop_rounding_dropped": ("if (hop) next_buffer[k] = round_to(next_buffer[k], dtype);", ";"),
    "f16_widen_subnormal": ("f = ldexpf((float)man, -24);", "f = ldexpf((float)man, -25);"),
    "sparse_threshold_inclusive": ("send[i] = fabsf(send[i]) > threshold ? send[i] : 0.0f;",
                                   "send[i] = fabsf(send[i]) >= threshold ? send[i] : 0.0f;"),
    "sparse_sort_ascending": ("if (x->key != y->key) return x->key > y->key ? -1 : 1;",
                              "if (x->key != y->key) return x->key < y->key ? -1 : 1;"),
    "sparse_k_floor": ("int64_t K = (int64_t)ceilf(threshold * (float)n);",
                       "int64_t K = (int64_t)floorf(threshold * (float)n);"),
    "sparse_residual_sign": ("for (int64_t i = 0; i < n; ++i) acc[i] = backup[i] - send[i];",
                             "for (int64_t i = 0; i < n; ++i) acc[i] = send[i] - backup[i];"),
    "sparse_rank_order": ("    for (int u = 0; u < W; ++u)\n      for (int64_t k = 0; k < len[u]; ++k)",
                          "    for (int u = W - 1; u >= 0; --u)\n      for (int64_t k = 0; k < len[u]; ++k)"),
    "sparse_index_base": ("result[lists[u][k].idx - 1] = 1.0f * lists[u][k].val + result[lists[u][k].idx - 1];",
                          "result[lists[u][k].idx % n] = 1.0f * lists[u][k].val + result[lists[u][k].idx % n];"),
    "sparse_tie_higher_index_first": ("return x->idx < y->idx ? -1 : (x->idx > y->idx ? 1 : 0);",
                                      "return x->idx > y->idx ? -1 : (x->idx < y->idx ? 1 : 0);"),
    "sparse_topk_residual_without_zero_scatter": (
        "for (int64_t k = 0; k < K; ++k) acc[lists[u][k].idx - 1] += 1.0f * lists[u][k].val;",
        "for (int64_t k = 0; k < K; ++k) acc[lists[u][k].idx - 1] = lists[u][k].val;"),
    "sparse_k_in_double": ("int64_t K = (int64_t)ceilf(threshold * (float)n);",
                           "int64_t K = (int64_t)ceil((double)threshold * (double)n);"),
    "bf16_nan_rounded_like_a_number": (
        "if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)\n",
        "if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0 && 0)\n"),
    "f16_nan_not_quieted": ("return (uint16_t)(sign | (man ? 0x7E00u | (man >> 13) : 0x7C00u));",
                            "return (uint16_t)(sign | (man ? 0x7C00u | (man >> 13) : 0x7C00u));"),
    "sampled_wrong_segment": ("if (idx[i] >= off && idx[i] < off + len) j = u;",
                              "if (idx[i] >= off && idx[i] < off + len) j = (u + 1) % W;"),
    "wire_avg_scales_unrounded_sum": ("if (hop) v = round_to(v, dtype);\n          if (op == ORACLE_AVG)",
                                      "if (0) v = round_to(v, dtype);\n          if (op == ORACLE_AVG)"),
    "allgatherv_block": ("int b = ufr[(W + p - s) % W]; /* block held at step s */",
                         "int b = ufr[(W + p + s) % W]; /* block held at step s */"),
    "allgatherv_displacement": ("char* dst = (char*)out[me] + disp[b] * es;",
                                "char* dst = (char*)out[me] + disp[me] * es;"),
}

BATTERY = r"""
import sys, traceback
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import oracle
import test_oracle_pins as P
pins = [
    (P.test_ring_schedule_matches_nccl_page_table, ()),
    (P.test_ring_schedule_structure, (5,)),
    (P.test_segments_golden, ()),
    (P.test_ring_order_hand_derived, ()),
    (P.test_brute_force_tiny, (3, 5)),
    (P.test_brute_force_tiny, (4, 16)),
    (P.test_integer_valued_sums_exact, (7,)),
    (P.test_avg_power_of_two_exact, (3,)),
    (P.test_avg_scale_rounding_hand_derived, ()),
    (P.test_max_matches_numpy, (4,)),
    (P.test_max_signed_zero_and_nan, ()),
    (P.test_bf16_rne_golden, ()),
    (P.test_bf16_nan_stays_nan, ()),
    (P.test_bf16_allreduce_accumulates_in_fp32, ()),
    (P.test_allgather_of_reduce_scatter_is_allreduce, (3, 10, oracle.F32, "sum")),
    (P.test_allgather_is_concatenation, (5,)),
    (P.test_fuse_plan_golden, ()),
    (P.test_pack_is_concatenation_and_unpack_inverts, ()),
    (P.test_fusion_allreduce_integer_mean_exact, ()),
    (P.test_min_matches_numpy, (4,)),
    (P.test_min_signed_zero_and_nan, ()),
    (P.test_prod_ring_order_hand_derived, ()),
    (P.test_prod_of_small_integers_exact, (3,)),
    (P.test_allgatherv_is_concatenation, (3,)),
    (P.test_f16_rne_golden, ()),
    (P.test_f16_nan_stays_nan, ()),
    (P.test_f16_widening_matches_numpy_for_all_patterns, ()),
    (P.test_wire_hop_rounding_hand_derived, ()),
    (P.test_wire_integer_sums_exact, ("f16", 3)),
    (P.test_sampled_equals_full, (8, 1000, "sum", oracle.F32)),
    (P.test_sparse_allreduce_hand_derived, ()),
    (P.test_sparse_threshold_matches_dense_definition, (3, True)),
    (P.test_sparse_topk_matches_sorted_selection, (2, 0.05)),
    (P.test_sparse_topk_count_rounding, ()),
    (P.test_sparse_topk_ties_and_signed_zero_hand_derived, ()),
]
failed = []
with oracle.using({so!r}):
    for fn, args in pins:
        try:
            fn(*args)
        except Exception:
            failed.append(fn.__name__)
print("FAILED_PINS", failed)
sys.exit(0 if failed else 3)
"""


def _build(src_text, tmp_path):
    src = tmp_path / "oracle.c"
    so = tmp_path / "liboracle_variant.so"
    src.write_text(src_text)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(src), "-lm"], check=True)
    return str(so)


def _battery(so):
    code = BATTERY.format(root=ROOT, here=HERE, so=so)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=600)


def _source():
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        return f.read()


def test_unmodified_oracle_passes_battery(tmp_path):
    r = _battery(_build(_source(), tmp_path))
    assert r.returncode == 3, r.stdout + r.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    orig, repl = MUTANTS[name]
    text = _source()
    assert text.count(orig) == 1, f"mutation site for {name} not unique/present"
    r = _battery(_build(text.replace(orig, repl), tmp_path))
    assert r.returncode != 3, f"planted mistake {name} survived every pin:\n{r.stdout}"
