"""Planted mistakes: the oracle's pins must catch each one.

Every case below copies ``oracle/kvoracle.c`` to a temporary directory,
plants one plausible slip by a textual edit (a flipped sign, a wrong pair
partner, a wrong frequency exponent, another rounding rule, a dropped patch
term, ...), compiles the copy and runs the pins of ``test_oracle_pins`` on
it.  At least one pin has to fail.  The committed oracle itself is never
modified.  Every planted edit keeps all memory accesses in bounds.
"""
import os

import pytest

import oracle as O
from oracle import build as obuild
import test_oracle_cdc_pins as CDC
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(obuild.__file__), "kvoracle.c")

# (name, text to replace, replacement, which occurrence (0-based))
MUTANTS = [
    ("sin-sign", "y[j] = lo * c - hi * s;", "y[j] = lo * c + hi * s;", 0),
    ("reversed-direction", "double c = cos(a), s = sin(a);", "double c = cos(a), s = -sin(a);", 0),
    ("pair-partner", "double lo = x[j], hi = x[j + h];", "double lo = x[j], hi = x[(j + 1) % h + h];", 0),
    ("theta-exponent", "pow(base, -2.0 * (double)j / (double)d)", "pow(base, -1.0 * (double)j / (double)d)", 0),
    ("theta-index", "pow(base, -2.0 * (double)j / (double)d)", "pow(base, -2.0 * (double)(j + 1) / (double)d)", 0),
    ("round-truncates", "double n = rint(ldexp(a, -q));", "double n = floor(ldexp(a, -q));", 0),
    ("round-ties-away", "double n = rint(ldexp(a, -q));", "double n = round(ldexp(a, -q));", 0),
    ("double-rounding", "double a = fabs(v);", "double a = (double)(float)fabs(v);", 0),
    ("no-subnormals", "if (E < -126)\n        E = -126;", "if (E < -150)\n        E = -150;", 0),
    ("identity-lost", "if (delta == 0) {\n        memmove", "if (0) {\n        memmove", 0),
    ("splice-rotates-by-minus-delta", "nr + p * rw + h * rd, rd, delta,", "nr + p * rw + h * rd, rd, -delta,", 0),
    ("splice-reads-span", "slot_of(pool, bt, max_blocks, s_end[q] + k)", "slot_of(pool, bt, max_blocks, s_start[q] + k)", 0),
    ("stub-reversed", "stub_copy + ((int64_t)l * total_stub + stub_base + k) * cd",
     "stub_copy + ((int64_t)l * total_stub + stub_base + (n_r - 1 - k)) * cd", 0),
    ("forget-keeps-span", "seq_lens[q] = s_start[q];", "seq_lens[q] = s_end[q];", 0),
    ("relocate-reversed-chunk", "int64_t d = slot_of(dst, bt, max_blocks, chunk_dst_pos[c] + (t - tok_off[c]));",
     "int64_t d = slot_of(dst, bt, max_blocks, chunk_dst_pos[c] + (tok_off[c + 1] - 1 - t));", 0),
    ("patch-drops-last-rank", "for (int r = 0; r < pt->m; ++r)", "for (int r = 0; r < pt->m - 1; ++r)", 0),
    ("patch-wrong-v-index", "s += (double)u[r] * (double)v[r];", "s += (double)u[r] * (double)v[0];", 0),
    ("patch-token-index", "pt->u_chunk_tok[c] + (t - tok_off[c]) : t;", "pt->u_chunk_tok[c] + (t - tok_off[c]) : t - tok_off[c];", 0),
    ("u-map-drops-offset", "pt->u_chunk_tok[c] + (t - tok_off[c]) :", "pt->u_chunk_tok[c] :", 0),
    ("v-map-ignored", "pt->v_chunk ? pt->v_chunk[c] : c;", "c;", 0),
    ("fused-patch-rounds-twice", "kvo_round_bf16(ex[i] + patch_term(patch, 1, l,",
     "kvo_round_bf16(kvo_bf16_to_f64(kvo_round_bf16(ex[i])) + patch_term(patch, 1, l,", 0),
    ("relocate-ignores-copy-patch", "if (has_patch(patch, 0)) {\n                    for (int col = 0; col < cd; ++col)\n                        dc[col]",
     "if (0) {\n                    for (int col = 0; col < cd; ++col)\n                        dc[col]", 0),
    ("interleaved-partner", "double even = x[2 * j], odd = x[2 * j + 1];", "double even = x[2 * j], odd = x[(2 * j + 3) % d];", 0),
    ("interleaved-sin-sign", "y[2 * j] = even * c - odd * s;", "y[2 * j] = even * c + odd * s;", 0),
    ("composed-origin-position-zero", "cur[p].written = p;", "cur[p].written = 0;", 0),
    ("composed-stub-never-rotated", "rd, p - cur[p].written,", "rd, cur[p].src >= 0 ? p - cur[p].written : 0,", 0),
    ("composed-stub-rows-ignore-sequence", "if (i2 < i || (i2 == i && q2 < q))", "if (i2 < i)", 0),
    ("xxh-round-rotation", "acc = rotl64(acc, 31);", "acc = rotl64(acc, 33);", 0),
    ("xxh-prime", "#define XXP2 0xC2B2AE3D27D4EB4Full", "#define XXP2 0xC2B2AE3D27D4EB4Dull", 0),
    ("xxh-four-byte-tail", "acc = rotl64(acc, 23) * XXP2 + XXP3;", "acc = rotl64(acc, 21) * XXP2 + XXP3;", 0),
    ("xxh-no-length", "acc += (uint64_t)len;", "acc += 0;", 0),
    ("splitmix-counter-offset", "seed + (n + 1u) * 0x9E3779B97F4A7C15ull", "seed + n * 0x9E3779B97F4A7C15ull", 0),
    ("gear-no-shift", "acc = 2u * acc + kvo_splitmix64_at", "acc = acc + kvo_splitmix64_at", 1),
    ("gear-window-sum-no-shift", "acc = 2u * acc + kvo_splitmix64_at", "acc = acc + kvo_splitmix64_at", 0),
    ("cdc-threshold-flipped", "if (acc < threshold || i == b - 1)", "if (acc > threshold || i == b - 1)", 0),
    ("cdc-hash-not-reset-per-stream", "        uint64_t acc = 0;\n        int64_t start = a;",
     "        static uint64_t acc = 0;\n        int64_t start = a;", 0),
    ("fingerprint-from-stream-start", "tokens_xxh64(tokens + start, i + 1 - start, fp_seed)",
     "tokens_xxh64(tokens + a, i + 1 - a, fp_seed)", 0),
    ("token-bytes-big-endian", "buf[4 * i] = (uint8_t)v;", "buf[4 * i] = (uint8_t)(v >> 24);", 0),
]


def _pins():
    """The pins as (name, callable(oracle)), cheapest first."""
    golden = P._golden_rne()
    return [
        ("worked-values", lambda o: [P.test_round_bf16_worked_values(o, v, w) for v, w in golden]),
        ("double-rounding", P.test_round_bf16_is_not_double_rounding),
        ("torch-rne", P.test_round_bf16_matches_torch_on_fp32_inputs),
        ("delta-zero", P.test_delta_zero_is_the_identity_bitwise),
        ("pair-zero", P.test_pair_zero_is_a_plain_2d_rotation),
        ("one-hot", P.test_one_hot_pairing),
        ("complex", lambda o: P.test_rotation_is_complex_multiplication(o, 10000.0, 64)),
        ("frequencies", lambda o: P.test_frequencies_are_geometric(o, 10000.0, 64)),
        ("norms", P.test_pair_norms_are_preserved),
        ("fresh-position", P.test_fresh_position_equivalence),
        ("relocate-brute", lambda o: P.test_relocate_matches_brute_force(o, 2, 8, 16)),
        ("fused-patch", P.test_fused_patch_matches_independent_restatement),
        ("factor-maps", P.test_factor_maps_reuse_factors_kept_per_chunk),
        ("patch-matmul", P.test_standalone_patch_matches_numpy_matmul),
        ("one-hot-patch", P.test_rank_one_one_hot_patch_touches_one_value),
        ("splice-batch", P.test_splice_batch_of_sequences_with_gqa_heads),
        ("splice-forget", P.test_splice_forget_truncates_without_moving_data),
        ("splice-successive", P.test_successive_directives_round_between_calls),
        ("splice-brute", P.test_splice_brute_force_every_directive),
        ("interleaved-complex", lambda o: P.test_interleaved_rotation_is_complex_multiplication(o, 64)),
        ("interleaved-ops", P.test_interleaved_relocate_and_splice_match_the_restatement),
        ("composed-single", P.test_composed_single_directive_is_the_splice),
        ("composed-batch", P.test_composed_three_directives_batch_gqa),
        ("composed-brute", P.test_composed_brute_force_two_directives),
        ("xxh64-empty", CDC.test_xxh64_published_empty_input_value),
        ("splitmix64-outputs", CDC.test_splitmix64_published_first_outputs),
        ("xxh64-library", CDC.test_xxh64_matches_the_installed_library),
        ("gear-window", CDC.test_gear_hash_is_the_64_token_window_sum),
        ("cdc-tiling", CDC.test_chunks_tile_each_stream_and_fingerprints_name_their_tokens),
        ("cdc-content", CDC.test_chunk_ends_follow_content_not_offset),
        ("cdc-mean-length", CDC.test_threshold_sets_the_mean_chunk_length),
        ("cdc-extremes", CDC.test_threshold_extremes_and_capacity),
    ]


def _plant(text, old, new, occurrence):
    idx = -1
    for _ in range(occurrence + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"planting site not found: {old!r}"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _plant(src, old, new, occ)
    assert mutated != src
    path = tmp_path / "kvoracle_mutant.c"
    path.write_text(mutated)
    lib = obuild.build(str(path), str(tmp_path / "libkvoracle_mutant.so"))
    mutant = O.Oracle(lib)
    caught = []
    for pin, fn in _pins():
        try:
            fn(mutant)
        except AssertionError:
            caught.append(pin)
            break
    assert caught, f"no pin caught the planted mistake {name!r}"
