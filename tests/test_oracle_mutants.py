"""The pins are sensitive: plausible mistakes planted in a copy of the oracle
(compiled on the CPU, never shipped) must each make at least one pin fail.

Each mutant is the oracle's source with one textual change -- a dropped term,
a wrong order, a different rounding, a wrong index -- built into its own
library and swapped in for the duration of the check.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_formats as fmt
import test_oracle_em_combine as em
import test_oracle_routing as rt

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.cpp")

MUTANTS = {
    # slot ignores the tokens earlier source ranks sent to the same rank
    "slot_without_source_prefix": ("for (int p = 0; p < src; ++p) running[r]", "for (int p = 0; p < 0; ++p) running[r]"),
    # combine sums in descending rank order
    "combine_descending": ("for (int r = 0; r < R; ++r) {\n        int sl = L.slot[static_cast<size_t>(t) * R + r];\n        if (sl < 0) continue;\n        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;\n        acc",
                           "for (int r = R - 1; r >= 0; --r) {\n        int sl = L.slot[static_cast<size_t>(t) * R + r];\n        if (sl < 0) continue;\n        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;\n        acc"),
    # scale taken as amax times a rounded reciprocal
    "scale_by_reciprocal": ("float scale = a / 448.0f;", "float scale = a * (1.0f / 448.0f);"),
    # e4m3 ties rounded away from zero
    "e4m3_ties_away": ("(frac == 0.5 && std::fmod(fl, 2.0) != 0.0)", "(frac == 0.5)"),
    # duplicate experts of one token counted twice for its rank
    "rank_counted_per_entry": [("L->in_rank[static_cast<size_t>(t) * R + r] = 1;",
                                "L->in_rank[static_cast<size_t>(t) * R + r] += 1;"),
                               ("L->tokens_per_rank[static_cast<size_t>(src) * R + r] += 1;",
                                "L->tokens_per_rank[static_cast<size_t>(src) * R + r] += L->in_rank[static_cast<size_t>(t) * R + r];")],
    # low-latency combine in k-index order instead of ascending expert id
    "ll_combine_k_order": ("while (pos > 0 && topk_idx[static_cast<size_t>(t) * k + order[pos - 1]] > e)", "while (false)"),
    # bf16 rounding truncates
    "bf16_truncates": ("if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u))) keep += 1u;", ""),
    # e4m3 combine input used without its scale
    "fp8_combine_ignores_scale": ("return code_value * y_scales[row * (H / 128) + h / 128];", "return code_value;"),
    # e4m3 combine input scaled by the row's first group only
    "fp8_combine_first_group_scale": ("y_scales[row * (H / 128) + h / 128]", "y_scales[row * (H / 128)]"),
    # top-k weights summed in descending rank order
    "combined_weights_descending": ("for (int r = 0; r < R; ++r) {\n        int sl = L.slot[static_cast<size_t>(t) * R + r];\n        if (sl < 0) continue;\n        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;\n        wsum",
                                    "for (int r = R - 1; r >= 0; --r) {\n        int sl = L.slot[static_cast<size_t>(t) * R + r];\n        if (sl < 0) continue;\n        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;\n        wsum"),
    # expert groups not padded to the alignment
    "em_groups_unaligned": ("int padded = ((*count)[e] + align - 1) / align * align;", "int padded = (*count)[e];"),
    # expert-major rows handed out in (k-index, token) order
    "em_rows_k_major": ("for (int t = 0; t < s.T; ++t)\n    for (int j = 0; j < s.k; ++j) {\n      int64_t e = topk_idx[static_cast<size_t>(t) * s.k + j];\n      if (e < 0) continue;\n      rank_in_expert",
                        "for (int j = 0; j < s.k; ++j)\n    for (int t = 0; t < s.T; ++t) {\n      int64_t e = topk_idx[static_cast<size_t>(t) * s.k + j];\n      if (e < 0) continue;\n      rank_in_expert"),
    # expert-major scales stored row-major
    "em_scales_row_major": ("recv_scales[g * scales_ld + rw] = sc[g];", "recv_scales[rw * G + g] = sc[g];"),
    # expert-major row weight taken from the token's first entry
    "em_weight_first_entry": ("recv_weights[rw] = topk_weights[static_cast<size_t>(t) * k + j];",
                              "recv_weights[rw] = topk_weights[static_cast<size_t>(t) * k];"),
    # expert-major combine in k-index order
    "em_combine_k_order": ("for (; at > 0 && ids[by_expert[at - 1]] > ids[j]; --at)", "for (; false; --at)"),
    # local expert id off by one rank
    "local_id_wrong_rank": ("here ? static_cast<int>(e - r * s.El) : -1", "here ? static_cast<int>(e - (r > 0 ? r - 1 : 0) * s.El) : -1"),
}


def _pins(golden_dir):
    """Every pin, as (name, callable); a mutant must fail at least one."""
    calls = [
        ("e4m3 hand points", lambda: fmt.test_e4m3_hand_encoded_points(golden_dir)),
        ("bf16 hand points", lambda: fmt.test_bf16_hand_rounded_points(golden_dir)),
        ("e4m3 vs torch", fmt.test_e4m3_encode_all_bf16_patterns_vs_torch),
        ("layout hand", lambda: rt.test_layout_hand_worked(golden_dir)),
        ("dispatch/combine hand", lambda: rt.test_dispatch_combine_hand_worked(golden_dir)),
        ("combine order hand", lambda: rt.test_combine_order_hand_worked(golden_dir)),
        ("ll hand", lambda: rt.test_low_latency_hand_worked(golden_dir)),
        ("ll combine order hand", lambda: rt.test_ll_combine_order_hand_worked(golden_dir)),
        ("layout brute force", lambda: rt.test_layout_vs_sorted_pairs(120, 3, 12, 4, 0.2, 0.3)),
        ("dispatch permutation", lambda: rt.test_dispatch_permutation_and_rows(True)),
        ("quantiser", rt.test_quantize_round_trip_bound_and_nearest_code),
        ("combine closed form", lambda: rt.test_combine_identity_expert_closed_form(8, 64, 8)),
        ("ll brute force", lambda: rt.test_ll_slots_and_counts_vs_sort(0.3)),
        ("ll exact", rt.test_ll_combine_brute_force_exact),
        ("combine weights order hand", lambda: em.test_combine_weights_order_hand_worked(golden_dir)),
        ("combine weights undo dispatch", lambda: em.test_combine_weights_undo_dispatch(8, 64, 8, 0.2)),
        ("fp8 combine closed form", lambda: em.test_fp8_combine_power_of_two_scales_closed_form(8, 64, 8)),
        ("fp8 combine bound", em.test_fp8_combine_general_within_bound),
        ("em hand", lambda: em.test_em_layout_hand_worked(golden_dir)),
        ("em brute force", lambda: em.test_em_layout_vs_sorted_entries(96, 8, 64, 6, 0.05, 0.1, 4)),
        ("em rows", lambda: em.test_em_dispatch_rows_and_padding(True)),
        ("em combine order hand", lambda: em.test_em_combine_order_hand_worked(golden_dir)),
        ("em combine closed form", lambda: em.test_em_combine_identity_expert_closed_form(8, 64, 8, 16)),
    ]
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch, golden_dir):
    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
        src = src.replace(old, new)
    mutated = tmp_path / "ep_oracle.cpp"
    mutated.write_text(src)
    (tmp_path / "ep_oracle.h").write_text(open(SRC.replace(".cpp", ".h")).read())
    so = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(mutated)], check=True)
    real = oracle._load()
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    mutant = oracle._load()
    assert mutant is not real
    failed = []
    for pin, fn in _pins(golden_dir):
        try:
            fn()
        except (AssertionError, oracle.OracleError):
            failed.append(pin)
    assert failed, f"no pin caught the planted mistake {name}"
