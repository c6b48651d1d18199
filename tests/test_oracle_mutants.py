"""Plants plausible mistakes in a COPY of the oracle source, builds it, and
checks that at least one pin test fails for each — evidence that the pins
constrain every part of the oracle.  Nothing here touches a GPU."""
import os
import subprocess

import pytest

import oracle
import test_oracle_append_and_formula as T_app
import test_oracle_attention as T_att
import test_oracle_formats as T_fmt

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original fragment, mutated fragment, pin tests expected to catch it)
MUTANTS = [
    ("drop softmax scale", "s[i] = scale * acc;", "s[i] = acc;",
     [lambda: T_att.test_toy_incremental_step_equals_full_recompute(16)]),
    ("interleaved head map", "int hq = h * G + g;", "int hq = g * Hkv + h;",
     [T_att.test_scores_scale_and_head_mapping]),
    ("scores against V", "acc += qv[d] * K[(size_t)i * D + d];",
     "acc += qv[d] * V[(size_t)i * D + d];",
     [lambda: T_att.test_bruteforce_matches_sdpa(3, 4, 2, 8, 16, 40)]),
    ("offset from block index", "(t % block_size)) * D;", "(t / block_size)) * D;",
     [lambda: T_att.test_bruteforce_matches_sdpa(3, 4, 2, 8, 16, 40)]),
    ("no normalisation", "o[d] = acc / l;", "o[d] = acc;",
     [T_att.test_closed_forms]),
    ("K scale from V", "ks = k_scale[blk * Hkv + h];", "ks = v_scale[blk * Hkv + h];",
     [T_att.test_fp8_cache_is_dequantised_bytes_times_scale]),
    ("subnormal exponent", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);",
     [T_fmt.test_e4m3_all_codes_match_torch]),
    ("ties to odd", "(d == bestd && (code & 1) == 0)", "(d == bestd && (code & 1) == 1)",
     [T_fmt.test_e4m3_encoder_matches_torch_round_to_nearest_even]),
    ("merge weight sign", "double w = exp(lse - M);", "double w = exp(M - lse);",
     [T_att.test_merge_of_partials_equals_full]),
    ("lse sign", "lse_out[row * Hq + hq] = m + log(l);",
     "lse_out[row * Hq + hq] = m - log(l);",
     [T_att.test_merge_of_partials_equals_full]),
    ("fresh block test", "    if (off == 0) {\n      float amax", "    if (off == 1) {\n      float amax",
     [T_app.test_append_fp8_uses_block_scale_or_opens_block]),
    ("f16 exponent bias", "v = ldexp(1.0 + (double)m / 1024.0, e - 15);",
     "v = ldexp(1.0 + (double)m / 1024.0, e - 14);",
     [T_fmt.test_f16_all_codes_match_numpy]),
    ("causal limit off by one", "int hi = n - (nl - 1 - qi);", "int hi = n - (nl - qi);",
     [lambda: T_att.test_multi_query_matches_masked_sdpa(3, 2, 8, 2, 16, 16, 40),
      T_att.test_multi_query_toy_rows_of_full_masked_computation]),
    ("causal limit reversed", "int hi = n - (nl - 1 - qi);", "int hi = n - qi;",
     [T_att.test_multi_query_rows_are_single_queries_over_shorter_contexts]),
    ("window start off by one", "? hi - window : 0;", "? hi - window + 1 : 0;",
     [lambda: T_att.test_sliding_window_matches_band_masked_sdpa(2, 4, 6, 8, 1, 8, 4, 37),
      T_att.test_sliding_window_special_cases]),
    ("window gather ignores q_len",
     "if (window > 0 && t1 - (nl - 1) - window > t0) t0 = t1 - (nl - 1) - window;",
     "if (window > 0 && t1 - window > t0) t0 = t1 - window;",
     [lambda: T_att.test_sliding_window_matches_band_masked_sdpa(2, 4, 6, 8, 1, 8, 4, 37)]),
    ("query row ignores token", "size_t row = row0 + qi;",
     "size_t row = row0;",
     [lambda: T_att.test_multi_query_matches_masked_sdpa(2, 4, 8, 1, 8, 4, 37)]),
    ("prefill rows from the wrong offset", "const size_t row0 = q_start ? (size_t)q_start[b] : (size_t)b * q_len;",
     "const size_t row0 = q_start ? (size_t)q_start[b] * 0 : (size_t)b * q_len;",
     [T_att.test_prefill_matches_causal_sdpa_over_the_prompt]),
    # (mutants must not write outside the caller's arrays: they run in-process)
    ("prefill token count of the first sequence", "const int nl = q_start ? q_start[b + 1] - q_start[b] : q_len;",
     "const int nl = q_start ? q_start[1] - q_start[0] : q_len;",
     [T_att.test_prefill_matches_causal_sdpa_over_the_prompt]),
    ("calibration skips re-quantising", "          row[d] = oracle_e4m3_from_float(r);",
     "          (void)r;",
     [T_app.test_calibrated_append_scale_is_the_block_max_power_of_two_and_nothing_saturates]),
    ("calibration keeps the opener's scale", "      sc = cand;\n    }\n  }",
     "      (void)cand;\n    }\n  }",
     [T_app.test_calibrated_append_scale_is_the_block_max_power_of_two_and_nothing_saturates]),
    ("calibration scale off by a power of two", "  int k = (m <= 0.875f) ? e - 9 : e - 8;",
     "  int k = (m <= 0.875f) ? e - 8 : e - 7;",
     [T_app.test_calibrated_append_scale_is_the_block_max_power_of_two_and_nothing_saturates]),
    ("kv bytes drops the 2", "return 2.0 * num_layers", "return 1.0 * num_layers",
     [T_app.test_kv_bytes_formula_matches_pages]),
]


@pytest.mark.parametrize("name,orig,mut,tests", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, orig, mut, tests):
    with open(SRC) as f:
        src = f.read()
    assert src.count(orig) == 1, f"fragment for '{name}' not unique in oracle.c"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(orig, mut))
    so = tmp_path / "libmutant.so"
    subprocess.run(["cc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(so), "-lm"], check=True)
    import ctypes
    real = oracle.lib()
    mutant = ctypes.CDLL(str(so))
    for fn in ("oracle_f16_to_double", "oracle_bf16_to_double", "oracle_e4m3_to_double",
               "oracle_e4m3_from_float", "oracle_kv_bytes_per_token", "oracle_append",
               "oracle_append_calibrated",
               "oracle_decode", "oracle_decode_multi", "oracle_prefill", "oracle_merge",
               "oracle_num_threads"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = 0
    for t in tests:
        try:
            t()
        except (AssertionError, ValueError):
            caught += 1
    assert caught == len(tests), f"mutant '{name}' survived its pin tests"
