"""Mutation check of the oracle's pins: each case plants one plausible
mistake in a copy of oracle/ep_oracle.c (a dropped term, a wrong index, an
off-by-one, a transposed operand, a wrong rounding or constant), builds it,
and runs the oracle's pin tests (tests/test_oracle_*.py) against that build.
At least one pin must fail for every mutant; the unmodified source must
pass.  CPU only: nothing here touches a GPU or the product library."""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")
PIN_TESTS = [os.path.join(ROOT, "tests", f) for f in (
    "test_oracle_formats.py", "test_oracle_layout.py", "test_oracle_rank.py",
    "test_oracle_roundtrip.py")]

# name -> (text in ep_oracle.c, replacement, occurrence to replace (0-based))
MUTANTS = {
    # number formats
    "bf16_ties_away": ("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;",
                       "if (lo >= 0x8000u) hi += 1u;", 0),
    "e4m3_saturates_to_nan": ("if (a >= 448.0) return (uint8_t)(sign | 0x7e);",
                              "if (a >= 448.0) return (uint8_t)(sign | 0x7f);", 0),
    "e4m3_truncates": ("double q = nearbyint(a / step) * step;",
                       "double q = floor(a / step) * step;", 0),
    "e4m3_exponent_bias": ("((e + 7) << 3)", "((e + 8) << 3)", 0),
    "e4m3_decode_bias": ("ldexp((double)(8 + M), E - 10)", "ldexp((double)(8 + M), E - 9)", 0),
    "e4m3_subnormal_step": ("? ldexp(1.0, -9) : ldexp(1.0, ilogb(a) - 3)",
                            "? ldexp(1.0, -10) : ldexp(1.0, ilogb(a) - 3)", 0),
    # FP8 block quantisation
    "amax_floor_dropped": ("if (amax < 1e-4f) amax = 1e-4f;", "if (amax <= 0.0f) amax = 1e-30f;", 0),
    "amax_over_half_the_block": ("    for (int c = 0; c < BLOCK_CHANNELS; ++c) {\n      float a = fabsf(",
                                 "    for (int c = 0; c < BLOCK_CHANNELS / 2; ++c) {\n      float a = fabsf(", 0),
    "ue8m0_byte_one_low": ("scale_ue8m0[(int64_t)b * scale_stride] = (uint8_t)biased;",
                           "scale_ue8m0[(int64_t)b * scale_stride] = (uint8_t)(biased - 1u);", 0),
    "amax_infinity_not_capped": ("if (amax > FLT_MAX) amax = FLT_MAX;", "", 0),
    "fp32_scale_inverted": ("float scale = amax / 448.0f;", "float scale = 448.0f / amax;", 0),
    "fp32_max_240": ("float inv = 448.0f / amax;", "float inv = 240.0f / amax;", 0),
    "ue8m0_rounds_down": ("if (bits & 0x7fffffu) biased += 1u;", "", 0),
    "ue8m0_multiplier_sign": ("ldexpf(1.0f, 127 - (int)biased)", "ldexpf(1.0f, (int)biased - 127)", 0),
    "scales_row_major": ("scale_f32[(int64_t)b * scale_stride] = scale;",
                         "scale_f32[(int64_t)b] = scale;", 0),
    # layout
    "slot_rank_one_based": ("slot_rank[p] = num_tokens_per_expert[(int64_t)i * E + e];\n"
                            "        num_tokens_per_expert[(int64_t)i * E + e] += 1;",
                            "num_tokens_per_expert[(int64_t)i * E + e] += 1;\n"
                            "        slot_rank[p] = num_tokens_per_expert[(int64_t)i * E + e];", 0),
    "rank_of_expert_modulo": ("is_token_in_rank[((int64_t)i * T_r + t) * R + e / E_l] = 1;",
                              "is_token_in_rank[((int64_t)i * T_r + t) * R + e % R] = 1;", 0),
    "rank_counted_per_slot": ("is_token_in_rank[((int64_t)i * T_r + t) * R + e / E_l] = 1;",
                              "is_token_in_rank[((int64_t)i * T_r + t) * R + e / E_l] += 1;", 0),
    # notify
    "rank_prefix_exclusive": ("      run += num_tokens_per_rank[(int64_t)i * R + j];\n"
                              "      rank_prefix_matrix[(int64_t)i * R + j] = run;",
                              "      rank_prefix_matrix[(int64_t)i * R + j] = run;\n"
                              "      run += num_tokens_per_rank[(int64_t)i * R + j];", 0),
    "expert_prefix_inclusive": ("      expert_prefix[(int64_t)i * E + e] = run;\n"
                                "      run += num_tokens_per_expert[(int64_t)i * E + e];",
                                "      run += num_tokens_per_expert[(int64_t)i * E + e];\n"
                                "      expert_prefix[(int64_t)i * E + e] = run;", 0),
    "alignment_rounds_down": ("((run + a - 1) / a) * a", "(run / a) * a", 0),
    "expert_totals_row_dropped": ("    expert_prefix[(int64_t)R * E + e] = run;\n", "", 0),
    "psum_shifted_by_one": ("psum[(int64_t)r * (E_l + 1) + l + 1] = s;",
                            "psum[(int64_t)r * (E_l + 1) + l] = s;", 0),
    "psum_wrong_rank": ("s += num_recv_tokens_per_expert[(int64_t)r * E_l + l];",
                        "s += num_recv_tokens_per_expert[(int64_t)l];", 0),
    "worst_tokens_off_by_one": ("run > num_worst_tokens", "run >= num_worst_tokens", 0),
    "worst_tokens_check_dropped": (
        "if (num_worst_tokens >= 0 && run > num_worst_tokens) rc = ORACLE_ERR_CAPACITY;",
        "if (num_worst_tokens >= 0 && run > num_worst_tokens) rc = ORACLE_OK;", 0),
    # normal dispatch
    "dispatch_drops_source_offset": (
        "psum[(int64_t)r * (E_l + 1) + l] + expert_prefix[(int64_t)i * E + e] + slot_rank[p];",
        "psum[(int64_t)r * (E_l + 1) + l] + slot_rank[p];", 0),
    "dispatch_local_index_transposed": ("int l = (int)(e % E_l);", "int l = (int)(e / R);", 0),
    "dispatch_src_idx_local": ("recv_src_idx[flat] = i * T_r + t;", "recv_src_idx[flat] = t;", 0),
    "dispatch_combine_idx_without_rank": ("combine_idx[p] = (int32_t)flat;",
                                          "combine_idx[p] = (int32_t)row;", 0),
    "dispatch_scales_without_rank": ("(int64_t)r * nb * cap_rows + row, cap_rows);",
                                     "row, cap_rows);", 0),
    "dispatch_capacity_not_reported": (
        "          combine_idx[p] = -1;\n          rc = ORACLE_ERR_CAPACITY;\n          continue;",
        "          combine_idx[p] = -1;\n          continue;", 0),
    # low-latency dispatch
    "ll_recv_count_exclusive": ("recv_count[e] = eprefix[(int64_t)R * E + e];",
                                "recv_count[e] = eprefix[(int64_t)(R - 1) * E + e];", 0),
    "ll_range_fields_swapped": (
        "((int64_t)eprefix[(int64_t)i * E + e] << 32) | (int64_t)ntpe[(int64_t)i * E + e];",
        "((int64_t)ntpe[(int64_t)i * E + e] << 32) | (int64_t)eprefix[(int64_t)i * E + e];", 0),
    "ll_max_tokens_check_dropped": ("if (R <= 0 || E % R != 0 || T_r > max_tokens_per_rank ||",
                                    "if (R <= 0 || E % R != 0 ||", 0),
    "ll_row_drops_source_offset": ("int64_t row = (int64_t)eprefix[(int64_t)i * E + e] + slot_rank[p];",
                                   "int64_t row = (int64_t)slot_rank[p];", 0),
    "ll_src_info_local": ("packed_recv_src_info[flat] = i * T_r + t;",
                          "packed_recv_src_info[flat] = t;", 0),
    "ll_combine_idx_without_expert": ("combine_idx[p] = (int32_t)flat;",
                                      "combine_idx[p] = (int32_t)row;", 1),
    "ll_scales_row_major": ("e * nb * seg_rows + row, seg_rows);",
                            "(e * seg_rows + row) * nb, 1);", 0),
    # combine
    "combine_weight_of_slot0": ("acc = fmaf(topk_weights[t * k + j],", "acc = fmaf(topk_weights[t * k],", 0),
    "combine_starts_from_minus_zero": ("      float acc = 0.0f;\n      for (int j = 0; j < k; ++j) {\n        int32_t f = combine_idx[t * k + j];\n        if (f < 0) continue;\n        acc = fmaf(",
                                       "      float acc = -0.0f;\n      for (int j = 0; j < k; ++j) {\n        int32_t f = combine_idx[t * k + j];\n        if (f < 0) continue;\n        acc = fmaf(", 0),
    "combine_weight_dropped": ("acc = fmaf(topk_weights[t * k + j], ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]), acc);",
                               "acc = acc + ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]);", 0),
    # once-per-rank layout and combine
    "rank_prefix_transposed": ("before += cnt[(int64_t)i * R + r];", "before += cnt[(int64_t)r * R + i];", 0),
    "rank_capacity_not_reported": (
        "          combine_idx[base + first] = -1;\n          rc = ORACLE_ERR_CAPACITY;",
        "          combine_idx[base + first] = -1;", 0),
    "rank_topk_global_index": ("recv_topk_idx[flat * k + j] = on_r ? e - (int64_t)r * E_l : -1;",
                               "recv_topk_idx[flat * k + j] = on_r ? e : -1;", 0),
    "rank_first_slot_is_last": ("            first = j;\n            break;", "            first = j;", 0),
    "rank_src_idx_local": ("recv_src_idx[flat] = i * T_r + t;", "recv_src_idx[flat] = t;", 1),
    "rank_topk_weight_dropped": ("on_r ? topk_weights[base + j] : 0.0f;", "on_r ? 1.0f : 0.0f;", 0),
    "rank_combine_keeps_last": ("acc = acc + ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]);",
                                "acc = ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]);", 0),
}


def _mutate(src: str, old: str, new: str, occ: int) -> str:
    pos = -1
    for _ in range(occ + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {old[:60]!r}"
    return src[:pos] + new + src[pos + len(old):]


def _build(src_text: str, out_dir: str, name: str) -> str:
    c = os.path.join(out_dir, f"{name}.c")
    so = os.path.join(out_dir, f"lib_{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", so, c, "-lm"])
    return so


def _run_pins(so: str) -> int:
    env = dict(os.environ, EP_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return r.returncode


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("oracle_mutants"))
    with open(SRC) as f:
        src = f.read()
    libs = {"unmodified": _build(src, out, "unmodified")}
    for name, (old, new, occ) in MUTANTS.items():
        libs[name] = _build(_mutate(src, old, new, occ), out, name)
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        codes = dict(zip(libs, ex.map(_run_pins, libs.values())))
    return codes


def test_unmodified_oracle_passes_its_pins(results):
    assert results["unmodified"] == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(results, name):
    # exit status 1: a pin failed (not a crash, a collection or a usage error)
    assert results[name] == 1, f"no pin fails for the planted mistake {name!r}: {results[name]}"
