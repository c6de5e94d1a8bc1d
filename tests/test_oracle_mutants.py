"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is a textual edit of oracle/moe_oracle.c compiled into a temporary
directory; the pins run against it in a child process (a mutant may crash).
CPU only. The real oracle is never modified.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("drop_b1", "h[f] = moe_oracle_gelu(acc + (double)b1e[f]);", "h[f] = moe_oracle_gelu(acc);"),
    ("drop_b2", "out[o] = acc + (double)b2e[o];", "out[o] = acc;"),
    ("gelu_sign", "0.5 * u * (1.0 + erf(u / sqrt(2.0)))", "0.5 * u * (1.0 - erf(u / sqrt(2.0)))"),
    ("gelu_tanh", "0.5 * u * (1.0 + erf(u / sqrt(2.0)))",
     "0.5 * u * (1.0 + tanh(0.7978845608028654 * (u + 0.044715 * u * u * u)))"),
    ("gelu_no_sqrt2", "erf(u / sqrt(2.0))", "erf(u)"),
    ("w1_row_for_all", "acc += (double)w1e[f * d + i] * (double)xrow[i];",
     "acc += (double)w1e[i] * (double)xrow[i];"),
    ("w2_transposed_square", "acc += (double)w2e[o * d_ff + f] * h[f];",
     "acc += (double)w2e[(f % d) * d_ff + (o % d_ff)] * h[f];"),
    ("router_drops_bias", "if (router_bias) acc += (double)router_bias[e];", ""),
    ("router_token0", "acc += (double)x[t * d + i] * (double)w_g[(int64_t)e * d + i];",
     "acc += (double)x[i] * (double)w_g[(int64_t)e * d + i];"),
    ("softmax_no_norm", "probs[t * N + e] = exp(l[e] - m) / s;", "probs[t * N + e] = exp(l[e] - m);"),
    ("topk_smallest", "if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] < l[best]) best = e;"),
    ("topk_tie_high", "if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("gates_not_renormalised", "gate[t * k + j] = score[t * k + j] / s;", "gate[t * k + j] = score[t * k + j];"),
    ("capacity_no_k", "ceil(cf * (double)(T * (int64_t)k) / (double)N)", "ceil(cf * (double)T / (double)N)"),
    ("capacity_floor", "double c = ceil(", "double c = floor("),
    ("capacity_keeps_lowest", "if (a->score > b->score) return -1;\n  if (a->score < b->score) return 1;",
     "if (a->score > b->score) return 1;\n  if (a->score < b->score) return -1;"),
    ("capacity_tie_high_token", "if (a->t < b->t) return -1;\n  if (a->t > b->t) return 1;\n  return 0;\n}\n\nstatic",
     "if (a->t < b->t) return 1;\n  if (a->t > b->t) return -1;\n  return 0;\n}\n\nstatic"),
    ("capacity_off_by_one", "int64_t keep = n < C ? n : C;\n    for (int64_t r = keep; r < n; ++r) slot",
     "int64_t keep = n < C ? n : C + 1 > n ? n : C + 1;\n    for (int64_t r = keep; r < n; ++r) slot"),
    ("slots_descending", "return (a->t > b->t) - (a->t < b->t);", "return (a->t < b->t) - (a->t > b->t);"),
    ("dropped_still_combined", "if (slot[t * k + j] < 0) continue;\n    int64_t e", "int64_t e"),
    ("combine_unweighted", "double w = gate[t * k + j];", "double w = 1.0;"),
    ("combine_squared_gate", "double w = gate[t * k + j];", "double w = gate[t * k + j] * gate[t * k + j];"),
    ("renorm_ignored", "if (flags & ORACLE_FLAG_RENORM_SURVIVORS) w = w / kept_sum;", ""),
    ("fallback_ignored", "if (kept == 0 && (flags & ORACLE_FLAG_IDENTITY_FALLBACK))", "if (0)"),
    ("stats_f_over_T", "f[e] /= (double)(T * k);", "f[e] /= (double)T;"),
    ("zloss_not_squared", "z += lse * lse;", "z += lse;"),
    ("expert_choice_lowest", "for (int64_t r = 0; r < keep; ++r) taken[req[r].t * N + e] = 1;",
     "for (int64_t r = 0; r < keep; ++r) taken[req[T - 1 - r].t * N + e] = 1;"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation site of {name} not found"
    mutated = src.replace(orig, planted, 1)
    msrc = tmp_path / "moe_oracle_mutant.c"
    msrc.write_text(mutated)
    lib = str(tmp_path / "libmutant.so")
    O.compile_oracle(str(msrc), lib)
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "oracle_pins.py"), lib],
                          capture_output=True, text=True, timeout=300, cwd=ROOT)
    if proc.returncode < 0:
        return  # the mutant crashed the pin run (killed by a signal): caught
    assert proc.returncode == 0, proc.stderr[-2000:]
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught the planted mistake {name}"


def test_pin_script_is_clean_on_the_real_oracle():
    """The child-process pin run reports no failure for the unmodified oracle,
    so a caught mutant is caught by its planted mistake alone."""
    lib = O.load().path
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "oracle_pins.py"), lib],
                          capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr[-2000:]
    assert json.loads(proc.stdout.strip().splitlines()[-1]) == []
