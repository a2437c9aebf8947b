"""Plant plausible mistakes in copies of the oracle and check that a pin catches each.

Every mutant is the oracle's C source with one edit (a dropped term, a wrong
sign, a wrong index, a swapped operand), compiled on the CPU into a temporary
directory.  The pins of test_oracle.py run against it; at least one of them
must fail.  The oracle itself is never modified.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

MUTANTS = {
    "rope_sign": ("x[i] = a * c - b * s;", "x[i] = a * c + b * s;"),
    "rope_freq": ("pow(theta, -2.0 * (double)i / (double)D)",
                  "pow(theta, -1.0 * (double)i / (double)D)"),
    "rope_pairing": ("double a = x[i], b = x[i + half];", "double a = x[i], b = x[half - 1 - i];"),
    "gqa_map": ("const int32_t kvh = h / group;", "const int32_t kvh = h % Hk;"),
    "causal_off_by_one": ("if (causal && j > qpos)", "if (causal && j >= qpos)"),
    "query_alignment": ("const int64_t qpos = L - qo_len + (t - qo_indptr[b]);",
                        "const int64_t qpos = (t - qo_indptr[b]);"),
    "page_offset": ("const int64_t page = indices[indptr[b] + j / P];\n"
                    "        const int64_t off = kv_off(page, kvh, j % P, Hk, P, D, nhd);\n"
                    "        for (int32_t d = 0; d < D; ++d) kv[d]",
                    "const int64_t page = indices[j / P];\n"
                    "        const int64_t off = kv_off(page, kvh, j % P, Hk, P, D, nhd);\n"
                    "        for (int32_t d = 0; d < D; ++d) kv[d]"),
    "head_page_layout": ("return ((page * Hk + h) * P + t) * (int64_t)D;",
                         "return ((page * P + t) * Hk + h) * (int64_t)D;"),
    "nhd_layout": ("if (nhd) return ((page * P + t) * Hk + h) * (int64_t)D;",
                   "if (nhd) return ((page * Hk + h) * P + t) * (int64_t)D;"),
    "last_page_len": ("return (n - 1) * page_size + last_page_len[b];", "return n * page_size;"),
    "lse_drops_max": ("const double l = m + log(sum);", "const double l = log(sum);"),
    "scale_dropped": ("scores[j] = sm_scale * dot;", "scores[j] = dot;"),
    "v_reads_k": ("o[d] += p * kv_elem(v_pages, kv_fp8, v_scale, off + d);",
                  "o[d] += p * kv_elem(k_pages, kv_fp8, v_scale, off + d);"),
    "merge_weight": ("wb * o_b[r * D + d]", "wa * o_b[r * D + d]"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "window_off_by_one": ("j < qpos - window_left + 1)", "j < qpos - window_left)"),
    "window_from_end": ("j < qpos - window_left + 1)", "j < L - window_left)"),
    "page_pos_keys_ignored": ("const int64_t kpos = page_pos ? (int64_t)page_pos[indptr[b] + j / P] + j % P : j;",
                              "const int64_t kpos = j;"),
    "page_pos_query_ignored": ("      if (rope_theta > 0.0) rope_rotate(qv, D, (double)qlog, rope_theta);",
                               "      if (rope_theta > 0.0) rope_rotate(qv, D, (double)qpos, rope_theta);"),
    "kv8_v_scale": ("o[d] += p * kv_elem(v_pages, kv_fp8, v_scale, off + d);",
                    "o[d] += p * kv_elem(v_pages, kv_fp8, k_scale, off + d);"),
    "merge_lse": ("const double l = M + log(exp(a - M) + exp(b - M));",
                  "const double l = M + log(exp(a - M) + exp(b - M) + 1.0);"),
    "append_pos": ("const int64_t pos = L - n_new + i;", "const int64_t pos = L - n_new + i - 1;"),
    "append_head": ("const int64_t src = (src_tok * Hk + h) * (int64_t)D;",
                    "const int64_t src = (src_tok * Hk + (Hk - 1 - h)) * (int64_t)D;"),
}


def _checks():
    c = []
    for kw in ([dict(), dict(rope_theta=10000.0), dict(qo_lens=[1, 3, 5, 2], causal=True),
                dict(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=500.0),
                dict(Hq=6, Hk=3, D=6, P=3)]):
        c.append(lambda kw=kw: pins.test_matches_dense_torch(kw))
    c += [pins.test_closed_form_single_key, lambda: pins.test_closed_form_zero_query(16),
          pins.test_closed_form_equal_keys, pins.test_empty_request,
          lambda: pins.test_page_size_and_contiguous_invariance(dict()),
          pins.test_dropping_pages_equals_masking, lambda: pins.test_split_merge_equals_unsplit(3),
          pins.test_merge_with_empty_state_is_identity, pins.test_merge_matches_logsumexp_of_union,
          pins.test_cascade_equals_flat, pins.test_rope_matches_complex_rotation,
          pins.test_rope_d2_is_rotation_by_position_radians,
          pins.test_causal_row_equals_decode_at_shorter_length,
          pins.test_append_then_attend_equals_concatenation,
          pins.test_kv_len_and_malformed_tables,
          pins.test_e4m3_decoder_matches_torch_and_closed_forms,
          lambda: pins.test_kv8_equals_attention_over_the_decoded_values(dict()),
          pins.test_kv8_scales_apply_to_keys_and_values,
          pins.test_window_of_one_sees_only_its_own_key,
          lambda: pins.test_window_equals_masking_older_keys(5),
          pins.test_window_causal_rows_equal_decode_with_window,
          lambda: pins.test_page_positions_rotate_at_the_logical_positions(dict()),
          pins.test_page_positions_shift_invariance,
          pins.test_nhd_pages_equal_hnd_pages]
    return c


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutant {name} no longer applies"
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmp_path, "mutant.c")
    so_path = os.path.join(tmp_path, "mutant.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", c_path, "-o",
                    so_path, "-lm"], check=True)
    caught = 0
    with oracle._library(so_path):
        for check in _checks():
            try:
                check()
            except (AssertionError, ValueError):
                caught += 1
    assert caught >= 1, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_every_check():
    for check in _checks():
        check()
