"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/moe_oracle.c (on the CPU),
compiles it, runs every pin against it in a subprocess, and requires at least
one pin to fail.  The unmodified source must pass them all.  The planted
mistakes stay in bounds (no mutant reads or writes outside its arrays)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gate_up_swapped": ("double g = gu[c], u = gu[f + c];", "double g = gu[f + c], u = gu[c];"),
    "down_transposed": ("            y[c] += hr * (double)wrow[c];",
                        "            y[c] += hr * (double)Wd_e[(int64_t)c * f + r];"),
    "silu_is_sigmoid": ("h[c] = g / (1.0 + exp(-g)) * u;", "h[c] = 1.0 / (1.0 + exp(-g)) * u;"),
    "ties_to_higher_id": ("    if (a < b)\n        return 0;\n    return ia < ib;",
                          "    if (a < b)\n        return 0;\n    return ia > ib;"),
    "nan_ranks_first": ("        return bn;", "        return an;"),
    "renorm_dropped": ("        if (renorm)\n", "        if (0)\n"),
    "softmax_over_chosen_only": ("        for (int32_t e = 0; e < E; ++e)\n            Z += exp((double)L[e] - m);",
                                 "        for (int32_t j = 0; j < k; ++j)\n            Z += exp((double)L[idx[t * k + j]] - m);"),
    "dispatch_reverse_tokens": ("    for (int64_t t = 0; t < T; ++t) {\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx[t * k + j];",
                                "    for (int64_t t = T - 1; t >= 0; --t) {\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx[t * k + j];"),
    "combine_wrong_slot_weight": ("            int64_t e = idx[t * k + j];\n            double wj = w[t * k + j];",
                                  "            int64_t e = idx[t * k + j];\n            double wj = w[t * k + (k - 1 - j)];"),
    "forward_combine_wrong_slot": ("            double wj = scale_inputs ? 1.0 : w[t * k + j];",
                                   "            double wj = scale_inputs ? 1.0 : w[t * k + (k - 1 - j)];"),
    "input_scale_also_on_output": ("            double wj = scale_inputs ? 1.0 : w[t * k + j];",
                                   "            double wj = w[t * k + j];"),
    "input_scale_ignored": ("        row_scale[pos[q]] = scale_inputs ? w[q] : 1.0;",
                            "        row_scale[pos[q]] = 1.0;"),
    "bias_dropped": ("            if (bias)\n                s += (double)bias[e];", "            (void)bias;"),
    "batched_rows_one_expert": ("        int64_t e = expert[r];", "        int64_t e = expert[0];"),
    "combine_slot_order_reversed": ("            const double *yr = y_perm + (int64_t)pos[t * k + j] * d;",
                                    "            const double *yr = y_perm + (int64_t)pos[t * k + (k - 1 - j)] * d;"),
    "router_weight_transposed": ("s += (double)x[t * d + i] * (double)Wr[(int64_t)e * d + i];",
                                 "s += (double)x[t * d + i] * (double)Wr[(int64_t)i * E + e];"),
}


def _run(oracle_mod, src, tag):
    so = oracle_mod.build_from_source(src, tag)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "mutant_runner.py"), so],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_unmodified_oracle_passes_every_pin(oracle):
    assert _run(oracle, oracle.source(), "unmodified") == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle, name):
    find, repl = MUTANTS[name]
    src = oracle.source()
    assert src.count(find) == 1, f"mutation site not unique/present: {name}"
    failed = _run(oracle, src.replace(find, repl), name)
    assert failed, f"no pin caught the planted mistake '{name}'"
