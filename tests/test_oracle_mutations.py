"""Planted mistakes in the oracle, each caught by a pin.

Each case copies the oracle's C source, writes one plausible mistake into the
copy (a dropped term, a wrong constant, sign, index or order), compiles it
with the oracle's own compiler flags, binds it in place of the oracle, and
runs the pins (functions of the other test_oracle_*.py files) that guard that
part of the definition: at least one of them must fail.  A control case runs
every pin used here on an unmodified copy built the same way, so a failure
comes from the planted mistake and not from the harness.  CPU only."""
import ctypes
import importlib
import os

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "stv_oracle.c")

QUANT = "test_oracle_quant"
ATTN = "test_oracle_attention"
ACC = "test_oracle_accept_commit"
I4 = "test_oracle_int4"
KV2 = "test_oracle_k4v2"
LOOK = "test_oracle_lookup"

# name -> (text in stv_oracle.c, replacement, pins [(module, function, kwargs)])
MUTATIONS = {
    "fp16 conversion truncates": (
        "double r = rint(ldexp(a, 11 - e));", "double r = floor(ldexp(a, 11 - e));",
        [(QUANT, "test_double_to_half_matches_numpy_rounding", {})]),
    "3-bit scale max/3": (
        "orc_double_to_half(m / 4.0)", "orc_double_to_half(m / 3.0)",
        [(QUANT, "test_quantizer_scale_is_fp16_of_quarter_max", {}),
         (QUANT, "test_quantizer_exhaustive_against_brute_force", {"s_bits": 0x3C00})]),
    "3-bit code offset 3": (
        "rint(orc_half_to_double(x[i]) / sd) + 4.0", "rint(orc_half_to_double(x[i]) / sd) + 3.0",
        [(QUANT, "test_quantizer_exhaustive_against_brute_force", {"s_bits": 0x3C00})]),
    "3-bit ties rounded up": (
        "rint(orc_half_to_double(x[i]) / sd) + 4.0", "floor(orc_half_to_double(x[i]) / sd + 0.5) + 4.0",
        [(QUANT, "test_quantizer_exhaustive_against_brute_force", {"s_bits": 0x3C00})]),
    "3-bit clamp at 6": (
        "if (c > 7.0) c = 7.0;\n    codes[i]", "if (c > 6.0) c = 6.0;\n    codes[i]",
        [(QUANT, "test_quantizer_exhaustive_against_brute_force", {"s_bits": 0x3C00})]),
    "block: odd and even codes swap halves": (
        "*bit = ((i & 1) ? 16 : 0) + 3 * (m % 5) + b;", "*bit = ((i & 1) ? 0 : 16) + 3 * (m % 5) + b;",
        [(QUANT, "test_block_layout_against_hand_derived_words", {})]),
    "V codes block-major inside a tile": (
        "ch * 24 + ((slot % TILE_TOK) / 32) * 12", "ch * 12 + ((slot % TILE_TOK) / 32) * (HEAD_DIM * 12)",
        [(QUANT, "test_v_layout_against_hand_derived_positions", {})]),
    "V scales token-major inside a tile": (
        "g * (TILE_TOK * 2) + (slot % TILE_TOK) * 2", "(slot % TILE_TOK) * (N_GROUPS * 2) + g * 2",
        [(QUANT, "test_v_layout_against_hand_derived_positions", {})]),
    "int8 Q over 126": (
        "(int8_t)rint(127.0 * orc_half_to_double(q[c]) / m)", "(int8_t)rint(126.0 * orc_half_to_double(q[c]) / m)",
        [(QUANT, "test_int8_q_quantizer_exact", {})]),
    "int8 Q truncated": (
        "(int8_t)rint(127.0 * orc_half_to_double(q[c]) / m)", "(int8_t)trunc(127.0 * orc_half_to_double(q[c]) / m)",
        [(QUANT, "test_int8_q_quantizer_exact", {}), (QUANT, "test_int8_q_quantizer_ties_to_even", {})]),
    "int8 dots with code - 3": (
        "kv[g * GROUP + i] = (int8_t)((int)orc_block_code(w, i) - 4);",
        "kv[g * GROUP + i] = (int8_t)((int)orc_block_code(w, i) - 3);",
        [(ATTN, "test_int8_dots_match_big_integer_recomputation", {})]),
    "score scale 1/8": (
        "s /= 16.0;", "s /= 8.0;",
        [(ATTN, "test_attention_matches_dense_bruteforce", {"path": "exact", "seed": 0})]),
    "int8: group 0's scale for every group": (
        "s += sk[g] * (double)dots[g];", "s += sk[0] * (double)dots[g];",
        [(ATTN, "test_attention_matches_dense_bruteforce", {"path": "int8", "seed": 0})]),
    "int8: sQ dropped": (
        "s = (double)sq * s / 16.0;", "s = s / 16.0;",
        [(ATTN, "test_attention_matches_dense_bruteforce", {"path": "int8", "seed": 0})]),
    "mask: the next node is visible too": (
        "anc[i] = m;", "anc[i] = m | ((i + 1 < t) ? (1u << (i + 1)) : 0u);",
        [(ATTN, "test_attention_matches_dense_bruteforce", {"path": "exact", "seed": 0}),
         (ATTN, "test_chain_tree_equals_sequential_single_row_decodes", {"path": "exact"})]),
    "V read from the K half": (
        "rc = decode_row(cv, seq, keys[a], h, 1, vd);", "rc = decode_row(cv, seq, keys[a], h, 0, vd);",
        [(ATTN, "test_attention_matches_dense_bruteforce", {"path": "exact", "seed": 0})]),
    "softmax without the maximum": (
        "double p = exp(score[a] - smax);", "double p = exp(score[a]);",
        [(ATTN, "test_closed_form_huge_scores_stay_finite", {})]),
    "acceptance: edges judged alone": (
        "ok[i] = ok[parent[i]] && draft[i] == argmax[parent[i]];", "ok[i] = draft[i] == argmax[parent[i]];",
        [(ACC, "test_acceptance_all_5040_shapes", {})]),
    "acceptance: ties go to higher indices": (
        "better = cand[a] < best_path[a];", "better = cand[a] > best_path[a];",
        [(ACC, "test_acceptance_tie_break_prefers_lower_indices", {})]),
    "acceptance: bonus token from the root": (
        "out_ids[best_len - 1] = argmax[best];", "out_ids[best_len - 1] = argmax[0];",
        [(ACC, "test_acceptance_all_5040_shapes", {})]),
    "commit: every row gets the first row's K": (
        "memcpy(k_words(hb, slot, 0), kc[i], 96);", "memcpy(k_words(hb, slot, 0), kc[0], 96);",
        [(ACC, "test_commit_equals_repacking_committed_rows", {})]),
    "int4 scale max/8": (
        "orc_double_to_half(m / 7.0)", "orc_double_to_half(m / 8.0)",
        [(I4, "test_scale_closed_forms", {"m": 7.0, "s": 1.0})]),
    "int4 nibbles in natural order": (
        "static int i4_pos(int e) { return ((e & 1) ? 16 : 0) + 4 * (e >> 1); }",
        "static int i4_pos(int e) { return 4 * e; }",
        [(I4, "test_word_layout_hand_derived", {})]),
    "2-bit V tokens in natural order": (
        "static int v2_pos(int t) { return ((t & 1) ? 16 : 0) + 2 * (t >> 1); }",
        "static int v2_pos(int t) { return 2 * t; }",
        [(KV2, "test_words_hand_derived", {}), (KV2, "test_byte_positions_hand_derived", {})]),
    "4/2-bit: K at 3 bits": (
        "orc_quantize_group_bits(kr + g * GROUP, 4, &s, u);", "orc_quantize_group_bits(kr + g * GROUP, 3, &s, u);",
        [(KV2, "test_words_hand_derived", {}), (KV2, "test_byte_positions_hand_derived", {})]),
    "b-bit clamp one level high": (
        "if (c > h - 1.0) c = h - 1.0;", "if (c > h) c = h;",
        [(KV2, "test_codes_are_the_nearest_representable_value", {"bits": 2, "m": 1.0})]),
    "lookup: shortest length first": (
        "for (int L = max_len; L >= min_len; --L) {", "for (int L = min_len; L <= max_len; ++L) {",
        [(LOOK, "test_against_byte_string_search", {"alphabet": 2, "n": 40})]),
    "lookup: earliest occurrence": (
        "for (int64_t p = n - L - 1; p >= 0; --p) {", "for (int64_t p = 0; p <= n - L - 1; ++p) {",
        [(LOOK, "test_against_byte_string_search", {"alphabet": 2, "n": 40})]),
}


def build_copy(tmp_path, old=None, new=None):
    text = open(SRC).read()
    if old is not None:
        assert text.count(old) == 1, f"the planted mistake's site must occur once: {old!r}"
        text = text.replace(old, new)
    c = tmp_path / "stv_oracle_copy.c"
    c.write_text(text)
    so = tmp_path / "liboracle_copy.so"
    oracle.compile_c(str(c), str(so))
    return oracle.bind(ctypes.CDLL(str(so)))


def run_pin(lib, module, name, kwargs):
    """Run one pin against `lib`; True when it passes."""
    fn = getattr(importlib.import_module(module), name)
    saved = oracle._load()
    oracle._lib = lib
    try:
        fn(**kwargs)
        return True
    except (AssertionError, RuntimeError):
        return False
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(tmp_path, name):
    old, new, pins = MUTATIONS[name]
    lib = build_copy(tmp_path, old, new)
    results = [run_pin(lib, *pin) for pin in pins]
    assert not all(results), f"no pin caught the planted mistake: {name}"


def test_unplanted_copy_passes_every_pin(tmp_path):
    lib = build_copy(tmp_path)
    pins = {(m, f, tuple(sorted(k.items()))) for _, _, ps in MUTATIONS.values() for m, f, k in ps}
    for m, f, k in sorted(pins):
        assert run_pin(lib, m, f, dict(k)), f"{m}.{f}{dict(k)} fails on an unmodified copy"
