"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong or transposed index, a wrong rounding rule),
builds it on the CPU, and runs the oracle pin tests against that copy: at least
one pin must fail.  Nothing here touches a GPU."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")
PINS = ["tests/test_oracle_f16.py", "tests/test_oracle_q8_0.py", "tests/test_oracle_bf16.py",
        "tests/test_oracle_attention.py", "tests/test_oracle_plan_append.py",
        "tests/test_oracle_mq.py"]

MUTANTS = {
    "no_normalisation": ("for (int d = 0; d < D; ++d) o[d] /= l;", ""),
    "interleaved_gqa": ("int i = (int)(ig / n_q), g = (int)(ig % n_q), h = g / group;",
                        "int i = (int)(ig / n_q), g = (int)(ig % n_q), h = g % n_kv;"),
    "mq_interleaved_gqa": ("int j = (int)((x / n_q) % q_len), g = (int)(x % n_q), h = g / group;",
                           "int j = (int)((x / n_q) % q_len), g = (int)(x % n_q), h = g % n_kv;"),
    "slot_as_page": ("block_table[(int64_t)i * bt_stride + t / ORACLE_PAGE]",
                     "block_table[(int64_t)i * bt_stride + t % ORACLE_PAGE]"),
    "transposed_page_head": ("int64_t row = (page * n_kv + kvh) * ORACLE_PAGE + slot;",
                             "int64_t row = (kvh * n_kv + page) * ORACLE_PAGE + slot;"),
    "dropped_scale": ("s[t - t0] = scale * dot;", "s[t - t0] = dot;"),
    "dropped_q8_scale": ("return sc * (double)((const int8_t *)data)[row * D + d];",
                         "return (double)((const int8_t *)data)[row * D + d];"),
    "wrong_q8_block_index": ("scales[row * (D / ORACLE_QBLOCK) + d / ORACLE_QBLOCK]",
                             "scales[row * (D / ORACLE_QBLOCK) + d % (D / ORACLE_QBLOCK)]"),
    "softmax_sign": ("double p = exp(s[t - a] - m);", "double p = exp(m - s[t - a]);"),
    "ties_to_odd": ("double rem = n - whole;  /* exact */\n    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0))",
                    "double rem = n - whole;  /* exact */\n    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) == 0.0))"),
    "bf16_ties_to_odd": ("double rem = n - whole;\n    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0))",
                         "double rem = n - whole;\n    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) == 0.0))"),
    "ties_toward_plus_inf": ("return y < 0.0 ? -floor(-y + 0.5) : floor(y + 0.5);",
                             "return floor(y + 0.5);"),
    "q8_scale_126": ("float d = fdiv32(amax, 127.0f);", "float d = fdiv32(amax, 126.0f);"),
    "merge_sign": ("double w = exp2((double)m2[s] - M);", "double w = exp2(M - (double)m2[s]);"),
    "segment_start": ("int64_t a = (int64_t)n_kv * row_page_start[i] + h * npg, b = a + npg;",
                      "int64_t a = (int64_t)n_kv * row_page_start[i] + h, b = a + npg;"),
    "append_slot": ("int slot = pos % ORACLE_PAGE;", "int slot = L % ORACLE_PAGE;"),
    "aligned_chunk_end": ("hi[n] = base + h * npg + (q + 1) * npg / c;",
                          "hi[n] = base + h * npg + (q + 1) * npg / c + (q + 1 < c);"),
    "aligned_balance_bound": ("t1 = 11 * T / (10 * (int64_t)num_chunks);",
                              "t1 = 12 * T / (10 * (int64_t)num_chunks);"),
    "aligned_without_room": ("for (int64_t t = t0; t1 > t0 && t <= t1; ++t)",
                             "for (int64_t t = t0; t1 >= t0 && t <= t1; ++t)"),
    "aligned_group_size": ("int64_t m = t / npg;", "int64_t m = (t + npg - 1) / npg;"),
    "partial_base_e": ("double p = exp2(s[t - t0] - m);", "double p = exp(s[t - t0] - m);"),
    "bf16_eight_fraction_bits": ("ulp = ldexp(1.0, e - 8); /* 8 significant bits */",
                                 "ulp = ldexp(1.0, e - 9); /* 8 significant bits */"),
    "bf16_exponent_bias": ("mag = ldexp((double)(128 + frac), expo - 134);",
                           "mag = ldexp((double)(128 + frac), expo - 133);"),
    "mq_query_one_late": ("int P = L - q_len + j;", "int P = L - q_len + j + (j > 0);"),
    "mq_append_position": ("bt_stride, i, h, L - q_len + j, num_pages, k_data, v_data,",
                           "bt_stride, i, h, L - q_len + j - (j > 0), num_pages, k_data, v_data,"),
    "f32_neighbour_value": ("if (dtype == ORACLE_F32) return (double)((const float *)data)[row * D + d];",
                            "if (dtype == ORACLE_F32) return (double)((const float *)data)[row * D + (d ^ 1)];"),
    "f32_append_swaps_k_v": ("/* the fp32 values, unrounded */\n                memcpy((float *)k_data + row * D, kx,",
                             "/* the fp32 values, unrounded */\n                memcpy((float *)k_data + row * D, vx,"),
    "f32_mq_append_swaps_k_v": ("/* stored as given */\n        memcpy((float *)k_data + row * D, kx,",
                                "/* stored as given */\n        memcpy((float *)k_data + row * D, vx,"),
    "window_one_too_short": ("return window > 0 && L > window ? L - window : 0;",
                             "return window > 0 && L > window ? L - window + 1 : 0;"),
    "window_first_page_rounded_up": (
        "- window_start(L, window) / ORACLE_PAGE",
        "- (window_start(L, window) + ORACLE_PAGE - 1) / ORACLE_PAGE"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mut.c")
        so = os.path.join(tmp, "libmut.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", "-ffp-contract=off",
                        c, "-o", so, "-lm"], check=True)
        env = dict(os.environ, PKV_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            *PINS], cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
