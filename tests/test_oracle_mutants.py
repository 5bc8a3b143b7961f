"""The oracle pins are strong enough to catch plausible mistakes.

Each case compiles a copy of oracle/pkv_oracle.c with one deliberate slip
(a wrong or transposed index, a dropped term, a wrong bias or rounding rule),
swaps it in for the real oracle library, and runs every pin in
test_oracle_pins.py against it: at least one pin must fail.  CPU only; the
real oracle is untouched.
"""
import ctypes
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = [
    ("block index uses the offset", "int32_t blk = a->block_tables[(int64_t)s * a->MB + t / a->b];\n        if (blk < 0",
     "int32_t blk = a->block_tables[(int64_t)s * a->MB + t % a->b];\n        if (blk < 0"),
    ("offset off by one", "int off = t % a->b;\n        double dot",
     "int off = (t + 1) % a->b;\n        double dot"),
    ("GQA heads interleaved instead of grouped", "    int G = a->Hq / a->Hkv;\n    int h = i / G;\n    double* qrow",
     "    int G = a->Hq / a->Hkv;\n    int h = i % a->Hkv; (void)G;\n    double* qrow"),
    ("score scale dropped", "sc[t - t0] = a->scale * dot;", "sc[t - t0] = dot;"),
    ("normalised by length, not by the sum", "for (int d = 0; d < D; ++d) o[d] /= sum;\n        free(sc);\n    }\n    return status;\n}\n\n/* Paged prefill",
     "for (int d = 0; d < D; ++d) o[d] /= L;\n        free(sc);\n    }\n    return status;\n}\n\n/* Paged prefill"),
    ("pool rows and columns transposed", "return ((blk * Hkv + h) * (int64_t)b + off) * D + d;",
     "return ((blk * Hkv + h) * (int64_t)D + d) * b + off;"),
    ("value gathered from the key pool", "acc[d] += w[t - t0] * elem_to_double(a->v_pool,", "acc[d] += w[t - t0] * elem_to_double(a->k_pool,"),
    ("E4M3 subnormal exponent", "v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    ("E4M3 bias", "v = ldexp(1.0 + f / 8.0, e - 7);", "v = ldexp(1.0 + f / 8.0, e - 8);"),
    ("E4M3 ties to odd", "(err == best_err && (c & 1) == 0 && (best & 1) == 1)",
     "(err == best_err && (c & 1) == 1 && (best & 1) == 0)"),
    ("E4M3 no saturation", "if (a >= 448.0) return (uint8_t)(sign | 0x7e);", "if (a >= 480.0) return (uint8_t)(sign | 0x7f);"),
    ("bf16 bias", "v = ldexp(1.0 + f / 128.0, e - 127);", "v = ldexp(1.0 + f / 128.0, e - 126);"),
    ("f16 subnormal scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("merge drops the partition sums", "double w = lp * exp(m[r * NP + p] - M);", "double w = exp(m[r * NP + p] - M);"),
    ("partition max not rebased", "m_out[r] = m;\n        l_out[r] = sum;", "m_out[r] = 0.0;\n        l_out[r] = sum;"),
    ("append slot offset off by one", "int off = (int)(slot % b);", "int off = (int)((slot + 1) % b);"),
    ("append encodes with multiply-by-scale", "float kq = kx / k_scale;", "float kq = kx * k_scale;"),
    ("prefill mask drops the diagonal", "int nk = p + 1;                                      /* keys 0..p */",
     "int nk = p;"),
    ("prefill positions ignore the earlier context", "int p = seq_lens[s] - n + (tok - query_start[s]);",
     "int p = tok - query_start[s];"),
    ("prefill query row taken per sequence", "for (int d = 0; d < D; ++d) qrow[d] = elem_to_double(q, q_dtype, r * D + d);",
     "for (int d = 0; d < D; ++d) qrow[d] = elem_to_double(q, q_dtype, ((int64_t)s * Hq + i) * D + d);"),
    ("prefill GQA heads interleaved", "int tok = (int)(r / Hq), i = (int)(r % Hq), h = i / G;",
     "int tok = (int)(r / Hq), i = (int)(r % Hq), h = i % Hkv; (void)G;"),
    ("copy skips the value pool", "memmove((char*)v_pool + dst * block_bytes, (char*)v_pool + src * block_bytes, (size_t)block_bytes);",
     "(void)0;"),
]


def _pin_calls():
    calls = [
        (pins.test_f16_decode_all_codes_match_numpy, {}),
        (pins.test_bf16_decode_all_codes_match_torch, {}),
        (pins.test_e4m3_decode_all_codes_match_torch, {}),
        (pins.test_e4m3_encode_round_trip_every_finite_code, {}),
        (pins.test_e4m3_encode_ties_to_even_at_every_midpoint, {}),
        (pins.test_e4m3_encode_saturates, {}),
        (pins.test_e4m3_encode_matches_torch_inside_the_range, {}),
        (pins.test_decode_matches_50_digit_brute_force, {}),
        (pins.test_decode_invariant_under_block_relabelling, {}),
        (pins.test_closed_form_one_token_returns_its_value, {}),
        (pins.test_closed_form_identical_keys_give_mean_value, {}),
        (pins.test_closed_form_dominant_key_selects_its_value, {}),
        (pins.test_gqa_equal_queries_give_equal_rows_and_zero_length_gives_zeros, {}),
        (pins.test_oracle_rejects_out_of_pool_block_ids, {}),
        (pins.test_copy_blocks_copies_pairs_and_nothing_else, {}),
        (pins.test_prefill_of_single_tokens_equals_decode, {}),
        (pins.test_prefill_first_prompt_token_returns_its_value, {}),
        (pins.test_prefill_in_two_chunks_equals_one_pass, {}),
        (pins.test_prefill_matches_50_digit_brute_force, {}),
        (pins.test_prefill_invariant_under_block_relabelling, {}),
    ]
    for dt in ("f16", "bf16", "e4m3"):
        for G in (1, 4):
            calls.append((pins.test_decode_matches_contiguous_library_attention, {"dtype": dt, "G": G}))
        calls.append((pins.test_append_lands_at_the_mapped_slot_only, {"dtype": dt}))
        calls.append((pins.test_prefill_matches_contiguous_causal_library_attention, {"dtype": dt, "G": 4}))
    for P in (16, 32, 48, 512):
        calls.append((pins.test_partitioned_merge_equals_unsplit, {"P": P}))
    return calls


def test_unmutated_oracle_passes_every_pin_call():
    for fn, kw in _pin_calls():
        fn(**kw)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation anchor not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", str(path), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(str(so))))
    monkeypatch.setattr(oracle, "_TABLES", {})
    caught = []
    for fn, kw in _pin_calls():
        try:
            fn(**kw)
        except (Exception, pytest.fail.Exception):  # a pin rejected the mutant
            caught.append(fn.__name__)
    assert caught, f"no pin caught the mutant: {name}"
