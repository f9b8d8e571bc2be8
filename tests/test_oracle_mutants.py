"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/i8kv_oracle.c, builds it, and
runs the pin tests against that build in a child process; the run must fail.
The planted mistakes are the kind the pages warn about (a probability scale
applied to the wrong tokens, a scale dropped from the sum) and ordinary
indexing slips."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "i8kv_oracle.c")

MUTANTS = {
    # query head -> KV head mapping
    "gqa_modulo": ("const int kvh = h / G;\n      double* O = out + ((size_t)b * Hq + h) * D;\n"
                   "      for (int d = 0; d < D; ++d) O[d] = 0.0;\n      if (L <= 0) continue;\n      const int8_t* qv",
                   "const int kvh = h % Hkv;\n      double* O = out + ((size_t)b * Hq + h) * D;\n"
                   "      for (int d = 0; d < D; ++d) O[d] = 0.0;\n      if (L <= 0) continue;\n      const int8_t* qv"),
    # V scale not folded into the probabilities
    "drop_v_scale": ("W[t - t0] = R(P * (double)v_scale[s_index(blk, kvh, off, Hkv, bs)], fp32);",
                     "W[t - t0] = R(P, fp32);"),
    # missing 1/sqrt(d)
    "drop_softmax_scale": ("return R(s * c, fp32);", "return s;"),
    # rounding half away from zero
    "round_half_away": ("static inline double rne(double x) { return nearbyint(x); }",
                        "static inline double rne(double x) { return round(x); }"),
    # 16-token probability groups instead of the 32 one MMA consumes
    "group_of_16": ("for (int j0 = t0; j0 < t1; j0 += group) {", "for (int j0 = t0; j0 < t1; j0 += group / 2) {"),
    # log-sum-exp merge without the partition sums
    "merge_drops_l": ("double w = l_g[g] * exp(m_g[g] - M);", "double w = exp(m_g[g] - M);"),
    # online softmax forgets to rescale l
    "prefix_no_l_rescale": ("        l *= alpha;\n", "\n"),
    # causal mask off by one
    "causal_off_by_one": ("const int n_keys = history_len + j + 1;\n      const int kvh = h / G;\n      const int8_t* qv",
                          "const int n_keys = history_len + j;\n      const int kvh = h / G;\n      const int8_t* qv"),
    # K chunk layout with token and chunk swapped
    "k_layout_swap": ("return ((((size_t)blk * Hkv + h) * (D / 16) + d / 16) * bs + off) * 16 + (d % 16);",
                      "return ((((size_t)blk * Hkv + h) * bs + off) * (D / 16) + d / 16) * 16 + (d % 16);"),
    # int32 QK accumulation truncated to 16 bits
    "qk_acc_int16": ("acc += (int32_t)qv[d] * (int32_t)k_cache[k_index(blk, kvh, d, off, Hkv, D, bs)];",
                     "acc = (int16_t)(acc + (int32_t)qv[d] * (int32_t)k_cache[k_index(blk, kvh, d, off, Hkv, D, bs)]);"),
    # RoPE: sign of the sine term, cos/sin halves of the table row swapped
    "rope_sign": ("    x[i] = ac - bsn;\n", "    x[i] = ac + bsn;\n"),
    "rope_table_swap": ("float c = cs[i], s = cs[h + i];", "float c = cs[h + i], s = cs[i];"),
    # RMSNorm: sum instead of mean, eps dropped, weight reversed, the query
    # normalized with the key's weight, a left-to-right sum of squares
    "rms_no_mean": ("float mean = ss * (1.0f / (float)D);", "float mean = ss;"),
    "rms_no_eps": ("float var = mean + eps;", "float var = mean;"),
    "rms_weight_reversed": ("x[i] = t * bf16_to_f32(w[i]);", "x[i] = t * bf16_to_f32(w[D - 1 - i]);"),
    "q_norm_with_k_weight": ("qk_transform(q + row, D, q_norm_w, eps, cs, rd, x);",
                             "qk_transform(q + row, D, k_norm_w, eps, cs, rd, x);"),
    "rms_sequential_sum": ("  if (n == 1) return x[0] * x[0];\n",
                           "  if (n > 1) {\n    float acc = 0.0f;\n    for (int i = 0; i < n; ++i) acc += x[i] * x[i];\n"
                           "    return acc;\n  }\n  if (n == 1) return x[0] * x[0];\n"),
    # high-precision chunk: causal limit off by one, history K scaled by sV
    "bf16_prefix_causal": ("const int n_keys = history_len + j + 1;\n      const int kvh = h / G;\n      const uint16_t* qv",
                           "const int n_keys = history_len + j;\n      const int kvh = h / G;\n      const uint16_t* qv"),
    "bf16_prefix_k_scale": ("const double sc = (double)k_scale[s_index(blk, kvh, off, Hkv, bs)];\n          for (int d = 0; d < D; ++d) kx[d]",
                            "const double sc = (double)v_scale[s_index(blk, kvh, off, Hkv, bs)];\n          for (int d = 0; d < D; ++d) kx[d]"),
    # BF16-KV prefix comparison: causal limit off by one, query head -> KV head by modulo
    "bf16kv_prefix_causal": ("const int visible = history_len + j + 1;", "const int visible = history_len + j;"),
    "bf16kv_prefix_kv_head": ("const int kv_head = h / G;", "const int kv_head = h % Hkv;"),
    # K smoothing: K multiplied by s instead of 1/s; query head -> KV head by modulo
    "smooth_k_not_inverted": ("if (k_smooth) smooth_vec(x, D, k_smooth + (size_t)h * D, 1);",
                              "if (k_smooth) smooth_vec(x, D, k_smooth + (size_t)h * D, 0);"),
    "smooth_q_head_modulo": ("smooth_vec(x, D, k_smooth + (size_t)(h / (Hq / Hkv)) * D, 0);",
                             "smooth_vec(x, D, k_smooth + (size_t)(h % Hkv) * D, 0);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new), encoding="utf-8")
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-o", str(lib),
                    str(mut), "-lm"], check=True)
    env = dict(os.environ, I8KV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_quant.py", "tests/test_oracle_rope.py", "tests/test_oracle_bf16_prefix.py",
                        "tests/test_oracle_attention.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
