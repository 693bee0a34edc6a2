"""Plant mistakes in copies of the oracle and check that the pins catch each.

Every mutant below is a plausible slip (a dropped term, a wrong sign, a wrong
index, swapped strides, a wrong count).  The test rewrites the oracle's C
source in a temporary directory, builds it, and requires at least one pin in
tests/oracle_pins.py to fail on it.  Nothing here touches the real oracle."""
import os
import subprocess
import sys

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "drop_smoothing_term": ("*loss = (1.0 - a) * nll + a * smooth;", "*loss = (1.0 - a) * nll;"),
    "nll_sign": ("double nll = lse - x[y];", "double nll = lse + x[y];"),
    "no_max_shift_in_sum": ("        d += exp(x[j] - m);\n        S += x[j];\n    }\n    double lse",
                            "        d += exp(x[j]);\n        S += x[j];\n    }\n    double lse"),
    "smoothing_over_v_minus_1": ("+ a / (double)V; /* smoothed target */",
                                 "+ a / (double)(V - 1); /* smoothed target */"),
    "target_off_by_one": ("double q = (j == y ? 1.0 - a : 0.0) + a / (double)V; /* smoothed",
                          "double q = (j == y + 1 ? 1.0 - a : 0.0) + a / (double)V; /* smoothed"),
    "rows_in_wrong_order": ("        int64_t i = r / dim1, j = r % dim1;\n        int64_t y = targets[i * ts0 + j * ts1];\n        double* grow",
                            "        int64_t i = r % dim0, j = r / dim0;\n        int64_t y = targets[i * ts0 + j * ts1];\n        double* grow"),
    "count_includes_ignored": ("        if (y == ignore_idx) continue;\n        ++n;",
                               "        ++n;"),
    "mean_not_divided_by_n": ("g = (dloss ? dloss[0] : 1.0) / denom;",
                              "g = (dloss ? dloss[0] : 1.0);"),
    "ties_away_from_zero": ("double r = nearbyint(v / q) * q;", "double r = round(v / q) * q;"),
    "combine_skips_rescale": ("if (p[1] > 0.0) d += p[1] * exp(p[0] - m);",
                              "if (p[1] > 0.0) d += p[1];"),
    "grad_missing_scale": ("grad[j] = g * (exp(x[j] - lse) - q);", "grad[j] = exp(x[j] - lse) - q;"),
    "fp16_subnormal_decode": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "weighted_target_weight_dropped": ("*loss = (1.0 - a) * w[y] * (lse - x[y])",
                                       "*loss = (1.0 - a) * (lse - x[y])"),
    "linear_grad_weight_wrong_column": ("acc += dl[r * V + v] * oracle_decode(hidden, dtype, r * H + h);",
                                        "acc += dl[r * V + v] * oracle_decode(hidden, dtype, r * H + (H - 1 - h));"),
    "linear_logits_unrounded_grad": ("for (int64_t i = 0; i < N * V; ++i) dl[i] = oracle_round(dl[i], dtype);",
                                     "for (int64_t i = 0; i < N * V; ++i) dl[i] = dl[i] * 1.0000001;"),
    "weighted_mean_over_count": ("const double denom = class_weights ? wsum : (double)n;",
                                 "const double denom = (double)n;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    mpath = os.path.join(tmp_path, "mutant.c")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.build(force=True, src=mpath, out=os.path.join(tmp_path, "libm.so"))
    # Run the pins in a child process: a broken oracle may also crash.
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys, oracle\n"
        "from tests import oracle_pins\n"
        f"lib = oracle.load({so!r})\n"
        "caught = []\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin(lib)\n"
        "    except AssertionError:\n"
        "        caught.append(pin.__name__)\n"
        "print('CAUGHT', ' '.join(caught))\n"
    )
    res = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         timeout=600)
    caught = []
    for line in res.stdout.splitlines():
        if line.startswith("CAUGHT"):
            caught = line.split()[1:]
    assert caught, f"no pin caught mutant {name} (exit {res.returncode})"
