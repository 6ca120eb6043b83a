"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a temporary copy of ``oracle/gdn_oracle.c``
(on the CPU), rebuilds it there and runs ``test_oracle_pins.py`` against the
copy; the pin suites (scalar gate and per-channel KDA gate) have to fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "decay_missing_in_dot": ("S[(size_t)i * K + j] *= alpha;", "S[(size_t)i * K + j] *= 1.0;"),
    "outer_product_transposed": ("S[(size_t)i * K + j] += u_out[i] * khat[j];",
                                 "S[(size_t)i * K + j] += u_out[j % V] * khat[i % K];"),
    "correction_sign": ("u_out[i] = beta * (v[i] - d);", "u_out[i] = beta * (d - v[i]);"),
    "output_uses_key": ("o += S[(size_t)i * K + j] * qhat[j];", "o += S[(size_t)i * K + j] * khat[j];"),
    "dt_bias_sign": ("gdn_oracle_softplus(a + dt_bias)", "gdn_oracle_softplus(a - dt_bias)"),
    "A_log_not_exponentiated": ("double g = -exp(A_log) *", "double g = -A_log *"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-b));", "return 1.0 / (1.0 + exp(b));"),
    "eps_outside_sqrt": ("double norm = sqrt(ss + L2NORM_EPS);", "double norm = sqrt(ss) + L2NORM_EPS;"),
    "gqa_modulo": ("int hk = h / group;", "int hk = h % HK;"),
    "align_column_off_by_one": ("long col = (x - 1) / block_size;", "long col = x / block_size;"),
    "boundary_duplicates_final": ("for (long p = p0 + 1; p < p0 + n; ++p) {",
                                  "for (long p = p0 + 1; p <= p0 + n; ++p) {"),
    "replay_decays_after_write": (
        "double h = S[(size_t)i * K + j] * alpha[t];\n        S[(size_t)i * K + j] = h + ut[i] * kt[j];",
        "double h = S[(size_t)i * K + j];\n        S[(size_t)i * K + j] = (h + ut[i] * kt[j]) * alpha[t];"),
    "conv_window_off_by_one": ("for (int j = 0; j < SL; ++j) dst[j] = seq[ntok[w] + j];",
                               "for (int j = 0; j < SL; ++j) dst[j] = seq[ntok[w] + j - (j > 0)];"),
    "layer_group_ignored": ("int g = layer_group ? layer_group[l] : 0;", "int g = 0;"),
    "boundary_fold_reads_written_pool": (
        "memcpy(S, pools_in + l * pool_elems + ((size_t)src * HV + h) * VK,",
        "memcpy(S, pools_out + l * pool_elems + ((size_t)src * HV + h) * VK,"),
    "kda_decay_along_value_rows": (
        "for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= alpha[j];",
        "for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= alpha[i % K];"),
    "kda_replay_decay_along_value_rows": ("double h = S[(size_t)i * K + j] * at[j];",
                                          "double h = S[(size_t)i * K + j] * at[i % K];"),
    "kda_bias_per_head_not_channel": (
        "al[j] = gdn_oracle_decay(a[(size_t)t * K + j], A_log, dt_bias[j]);",
        "al[j] = gdn_oracle_decay(a[(size_t)t * K + j], A_log, dt_bias[0]);"),
    "kda_gate_ignores_head": ("memcpy(aa + (size_t)t * K, a + ((size_t)row * HV + h) * K,",
                              "memcpy(aa + (size_t)t * K, a + ((size_t)row * HV) * K,"),
    "kda_record_keeps_first_gate": (
        "memcpy(rec_g + rec * K, ga + (size_t)t * K, (size_t)K * sizeof(double));",
        "memcpy(rec_g + rec * K, ga, (size_t)K * sizeof(double));"),
    "source_one_token_late": (
        "int32_t s = slot_after(table_row, table_stride, block_size, seq_pos);",
        "int32_t s = slot_after(table_row, table_stride, block_size, seq_pos + 1);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "gdn_oracle.c")).read()
    assert before in src, f"mutation site for {name} not found"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    (tmp_path / "oracle" / "gdn_oracle.c").write_text(src.replace(before, after))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutants.py"))
    pkg = tmp_path / "spec_decode_recurrent_gb300"
    pkg.mkdir()
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "spec_decode_recurrent_gb300", f), pkg / f)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_kda_pins.py"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
