"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake (a dropped term, a wrong sign or index, a
transposed operand, an off-by-one) in a copy of the oracle's C source, builds
it with gcc in a temporary directory, and runs the oracle pin tests against
that copy in a subprocess: the run must fail.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "extkv_oracle.c")

MUTATIONS = {
    "gqa_head_map": ("int64_t kv = h / (Hq / Hkv);", "int64_t kv = h % Hkv;"),
    "scale_dropped": ("double t = scale * dot;", "double t = dot;"),
    "bias_dropped": ("s[j] = t + bj;", "s[j] = t;"),
    "softcap_after_bias": ("if (softcap > 0.0) t = softcap * tanh(t / softcap);\n    s[j] = t + bj;",
                           "s[j] = t + bj;\n    if (softcap > 0.0) s[j] = softcap * tanh(s[j] / softcap);"),
    "softcap_unscaled": ("t = softcap * tanh(t / softcap);", "t = tanh(t / softcap);"),
    "sentinel_inclusive": ("in_u[j] = (unsigned char)(!bias || bj > lowest);",
                           "in_u[j] = (unsigned char)(!bias || bj >= lowest);"),
    "window_off_by_one": ("p - j < window", "p - j <= window"),
    "offset_not_clamped": ("(np - S_q > 0 ? np - S_q : 0)", "(np - S_q)"),
    "softmax_sign": ("double w = exp(s[j] - m);", "double w = exp(m - s[j]);"),
    "v_reads_k": ("y[d] += w * orc_load(v_cache,", "y[d] += w * orc_load(k_cache,"),
    "span_end_inclusive": ("j >= lo && j < hi", "j >= lo && j <= hi"),
    "scatter_ignores_offset": ("* max_seq + (w + s)) * D + d;", "* max_seq + s) * D + d;"),
    "query_row_reversed": ("const int64_t q_off = ((b * Hq + h) * S_q + i) * Dk;",
                           "const int64_t q_off = ((b * Hq + h) * S_q + (S_q - 1 - i)) * Dk;"),
    "v_rows_with_key_stride": ("orc_load(v_cache, (kv_base + j) * Dv + d, dt)",
                               "orc_load(v_cache, (kv_base + j) * Dk + d, dt)"),
    "k_rows_with_value_stride": ("orc_load(k_cache, (kv_base + j) * Dk + d, dt)",
                                 "orc_load(k_cache, (kv_base + j) * Dv + d, dt)"),
    "causal_strict": ("int causal_ok = !causal || j <= p;", "int causal_ok = !causal || j < p;"),
    "padding_ignored_in_bias": ("if (j >= nonpad) return 0;", ""),
    "scatter_v_from_k": ("orc_copy_elem(v_cache, dst, v_new, src, dt);", "orc_copy_elem(v_cache, dst, k_new, src, dt);"),
    "q_start_ignored": ("int64_t qs = q_start ? q_start[b] : (np - S_q > 0 ? np - S_q : 0);",
                        "int64_t qs = (np - S_q > 0 ? np - S_q : 0);"),
    "denominator_counts_masked": ("    if (!in_u[j]) continue;\n    double w = exp(s[j] - m);\n    denom += w;",
                                  "    double w = in_u[j] ? exp(s[j] - m) : 0.0;\n    denom += in_u[j] ? w : 1.0;"),
    "bool_mask_inverted": ("if (mask[i]) orc_store_zero(bias, i, dt);", "if (!mask[i]) orc_store_zero(bias, i, dt);"),
    "extra_term_dropped": ("if (extra) orc_copy_elem(bias, idx, extra, idx, dt);",
                           "if (extra) orc_store_zero(bias, idx, dt);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                    str(mutant), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    tests = [os.path.join(ROOT, "tests", f) for f in
             ("test_oracle_bias.py", "test_oracle_scatter.py", "test_oracle_attention.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *tests], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the oracle pins:\n{r.stdout[-2000:]}"
