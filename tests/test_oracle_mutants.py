"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the oracle's C source (on the CPU, in a temporary
directory), builds it, and runs the pin suite against that build in a
subprocess: the suite has to fail."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pgd_oracle.c")

MUTANTS = {
    "sink_scaled": ("double sink = job->sinks ? (double)job->sinks[h] : -INFINITY;",
                    "double sink = job->sinks ? job->scale * (double)job->sinks[h] : -INFINITY;"),
    "group_modulo": ("int g = h / group;", "int g = h % job->kv_heads;"),
    "window_off_by_one": ("if (window > 0 && n - window + 1 > 0) lo = n - window + 1;",
                          "if (window > 0 && n - window > 0) lo = n - window;"),
    "sink_not_in_denominator": ("double z = (sink == -INFINITY) ? 0.0 : exp(sink - m);",
                                "double z = 0.0;"),
    "unscaled_scores": ("score[j] = scale * dot;", "score[j] = dot;"),
    "max_without_sink": ("double m = m_real > sink ? m_real : sink;", "double m = m_real;"),
    "slot_uses_quotient": ("slots[b] = (int64_t)page * page_size + n % page_size;",
                           "slots[b] = (int64_t)page * page_size + n / page_size;"),
    "gather_wrong_page_index": ("int64_t page_index = s / page_size;",
                                "int64_t page_index = s % page_size;"),
    "page_major_heads_swapped": (
        "return ((page * kv_heads + kv_head) * page_size + in_page) * head_dim + d;",
        "return ((kv_head * kv_heads + page) * page_size + in_page) * head_dim + d;"),
    "prefill_row_ignored": ("      trow = job->row_of[b];", "      trow = b;"),
    "rope_adjacent_pairs": ("const double b = bf16_value(xr[h * head_dim + i + half]);",
                            "const double b = bf16_value(xr[h * head_dim + (i ^ 1)]);"),
    "rope_sin_sign": ("orow[h * head_dim + i] = f64_to_bf16_rne(a * ci - b * si);",
                      "orow[h * head_dim + i] = f64_to_bf16_rne(a * ci + b * si);"),
    "rope_frequency_exponent": ("const float scaled = ((float)i * 2.0f) / (float)head_dim;",
                                "const float scaled = ((float)i * 1.0f) / (float)head_dim;"),
    "value_from_key": ("const uint16_t* vj = v + (int64_t)(lo + j) * head_dim;",
                       "const uint16_t* vj = k + (int64_t)(lo + j) * head_dim;"),
    "newest_key_dropped": ("int count = n - lo + 1;", "int count = n - lo;"),
    "weights_not_normalised": ("double p = exp(score[j] - m) / z;",
                               "double p = exp(score[j] - m);"),
    "kv_head_values_unstrided": ("v_rows + (int64_t)g * stride * d_head, n, d_head,",
                                 "v_rows + (int64_t)g * d_head, n, d_head,"),
    "lse_real_against_sink_max": ("z_real += exp(score[j] - m_real);",
                                  "z_real += exp(score[j] - m);"),
    "dense_rows_kv_heads_unstrided": (
        "k_rows = job->k + (int64_t)b * job->kv_heads * job->key_stride * d_head;",
        "k_rows = job->k + (int64_t)b * job->key_stride * d_head;"),
    "rope_angle_sin_cos_swapped": ("cos_out[i] = f64_to_bf16_rne(cos((double)angle));",
                                   "cos_out[i] = f64_to_bf16_rne(sin((double)angle));"),
    "head_major_head_stride": (
        "return ((int64_t)kv_head * num_pages * page_size + slot) * head_dim + d;",
        "return ((int64_t)kv_head * page_size + slot) * head_dim + d;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "libmutant.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so, c,
                        "-lm"], check=True)
        env = dict(os.environ, PGD_ORACLE_LIB=so)
        run = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                              os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                             cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert run.returncode != 0, f"mutant {name} passed every pin:\n{run.stdout[-2000:]}"
