"""The pins must be strong enough to catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle.c (on the CPU), builds it,
and runs the pin suite against it through ORACLE_LIB; the suite has to fail.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "causal_drops_diagonal": ("for (int j = 0; j <= i; ++j) {\n                z[j]",
                              "for (int j = 0; j < i; ++j) {\n                z[j]"),
    "unnormalised_rows": ("cu[j] += exp(z[j] - mi) / li;", "cu[j] += exp(z[j] - mi);"),
    "scale_dropped": ("z[j] = scale * dot(Qu", "z[j] = dot(Qu"),
    "q_k_transposed": ("dot(Qu + (size_t)i * d, Ku + (size_t)j * d, d)",
                       "dot(Qu + (size_t)j * d, Ku + (size_t)i * d, d)"),
    "topk_ties_to_higher": ("return (x->j < y->j) ? -1 : (x->j > y->j);",
                            "return (x->j > y->j) ? -1 : (x->j < y->j);"),
    "recent_window_short": ("for (int j = ncand; j < T; ++j) keep[j] = 1;",
                            "for (int j = ncand + 1; j < T; ++j) keep[j] = 1;"),
    "new_token_not_attended": ("for (int s = 0; s <= n; ++s) lsum += exp(z[s] - mx);\n        for (int e = 0; e < d; ++e) ou[e] = 0.0;\n        for (int s = 0; s <= n; ++s) {",
                               "for (int s = 0; s < n; ++s) lsum += exp(z[s] - mx);\n        for (int e = 0; e < d; ++e) ou[e] = 0.0;\n        for (int s = 0; s < n; ++s) {"),
    "window_boundary_off_by_one": ("if (ncand > 0 && !(pu[s] <= p - r)) continue;\n                if (best",
                                   "if (ncand > 0 && !(pu[s] < p - r)) continue;\n                if (best"),
    "evict_max_score": ("if (best < 0 || su[s] < su[best])", "if (best < 0 || su[s] > su[best])"),
    "no_accumulate": ("for (int s = 0; s < n; ++s) su[s] += exp(z[s] - mx) / lsum;",
                      "for (int s = 0; s < n; ++s) su[s] += 0.0;"),
    "new_score_zero": ("su[slot] = P_new;", "su[slot] = 0.0;"),
    "evict_ties_to_higher": ("if (best < 0 || su[s] < su[best])", "if (best < 0 || su[s] <= su[best])"),
    "lsh_zero_sets_bit": ("if (acc > 0.0f) code", "if (acc >= 0.0f) code"),
    "lsh_min_distance": ("if (dist > bestd) { bestd = dist; best = s; }",
                         "if (bestd < 0 || dist < bestd) { bestd = dist; best = s; }"),
    "lsh_ties_to_higher": ("if (dist > bestd) { bestd = dist; best = s; }",
                           "if (dist >= bestd) { bestd = dist; best = s; }"),
    "lsh_window_ignored": ("if (ncand > 0 && !(pos[s] <= p - r)) continue;", ""),
    "kv8_ties_away_from_zero": ("float y = rintf((float)x[e] * inv);", "float y = roundf((float)x[e] * inv);"),
    "kv8_scale_over_128": ("scale[t] = amax / 127.0f;", "scale[t] = amax / 128.0f;"),
    "kv8_inverse_from_128": ("float inv = 127.0f / amax;", "float inv = 128.0f / amax;"),
    "kv4_ties_away_from_zero": ("float y = rintf(inv * (float)x[e]);", "float y = roundf(inv * (float)x[e]);"),
    "kv4_product_in_fp64": ("float y = rintf(inv * (float)x[e]);", "float y = (float)rint((double)inv * x[e]);"),
    "kv4_scale_over_8": ("scale[t] = amax / 7.0f;", "scale[t] = amax / 8.0f;"),
    "kv4_inverse_from_8": ("float inv = 7.0f / amax;", "float inv = 8.0f / amax;"),
    "gqa_last_head_only": ("add[s] += P;                          /* heads in order g = 0..G-1 */",
                           "add[s] = P;"),
    "sh_threshold_share_of_n": ("const double t = P * (double)(n + 1);", "const double t = P * (double)n;"),
    "sh_prompt_threshold_share_of_i": ("exp(z[j] - mx) / l * (double)(i + 1);", "exp(z[j] - mx) / l * (double)i;"),
    "sh_flag_at_equal": ("const uint32_t f = t > 1.0 ? 1u : 0u;", "const uint32_t f = t >= 1.0 ? 1u : 0u;"),
    "sh_window_31": ("for (int b = 0; b < 32; ++b) n +=", "for (int b = 0; b < 31; ++b) n +="),
    "sh_evict_newest": ("if (a < b || (a == b && pu[s] < pu[best])) best = s;",
                        "if (a < b || (a == b && pu[s] > pu[best])) best = s;"),
    "sh_evict_most_pivotal": ("if (a < b || (a == b && pu[s] < pu[best])) best = s;",
                              "if (a > b || (a == b && pu[s] < pu[best])) best = s;"),
    "sh_select_ties_older": ("for (int j = ncand - 1; j >= 0; --j) {", "for (int j = 0; j < ncand; ++j) {"),
    "sh_prompt_rows_31": ("const int i0 = T > 32 ? T - 32 : 0;", "const int i0 = T > 31 ? T - 31 : 0;"),
    "sh_new_flag_dropped": ("else flag_new = f;", "else flag_new = 0u;"),
    "sh_history_not_shifted": ("if (s < n) mu[s] = (mu[s] << 1) | f;", "if (s < n) mu[s] = mu[s] | f;"),
    "fg_local_window_short": ("if (j >= i - B + 1) keep_l += a;", "if (j >= i - B + 2) keep_l += a;"),
    "fg_heavy_ignored": ("(heavy[j] && j <= i - r)) keep_f += a;", "(0 && heavy[j])) keep_f += a;"),
    "fg_frequency_first": ("policy[u] = rec_local[u] >= tau ? 0 : (rec_freq[u] >= tau ? 1 : 2);",
                           "policy[u] = rec_freq[u] >= tau ? 1 : (rec_local[u] >= tau ? 0 : 2);"),
    "fg_recovery_over_t_minus_1": ("rec_local[u] = keep_l / (double)T;", "rec_local[u] = keep_l / (double)(T - 1);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mutated = src.replace(old, new)
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "oracle_mut.c")
        so = os.path.join(tmp, "liboracle_mut.so")
        open(c, "w").write(mutated)
        subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
                        "-ffp-contract=off", c, "-o", so, "-lm"], check=True)
        env = dict(os.environ, ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
        assert r.returncode != 0, "planted mistake %s passed every pin:\n%s" % (name, r.stdout[-2000:])
