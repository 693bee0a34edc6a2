"""Values printed on the pages, checked against the oracle (CPU only).

Each fixture under tests/golden/ names its page and section and states the
reading taken of the printed example."""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_pitfall1_logsumexp_of_uniform_row_at_100(oracle_lib):
    g = _read("ops_nn_pitfall1_logsumexp.txt")
    V = int(g["V"])
    x = np.full((1, V), g["logit"], dtype=np.float32)
    r = oracle.ce(x, oracle.F32, 1, 1, V, targets=np.array([7]), want_grad=False, lib=oracle_lib)
    assert abs(r["lse"][0] - g["logsumexp"]) <= g["abs_tol"]
    assert abs(r["loss"][0] - g["loss"]) <= g["abs_tol"]
    assert np.isfinite(r["lse"][0])


def test_pitfall3_smoothing_share_of_gradient(oracle_lib):
    g = _read("ops_nn_pitfall3_smoothing_grad.txt")
    V = int(g["V"])
    x = np.zeros((1, V), dtype=np.float32)
    t = np.array([11])
    g0 = oracle.ce(x, oracle.F32, 1, 1, V, targets=t, lib=oracle_lib)["grad"][0]
    ga = oracle.ce(x, oracle.F32, 1, 1, V, targets=t, label_smoothing=g["label_smoothing"],
                   lib=oracle_lib)["grad"][0]
    share = g0[0] - ga[0]   # what smoothing subtracts from an off-target class
    assert abs(share - g["smoothing_share"]) <= g["rel_tol"] * g["smoothing_share"]
    # the target class gets back (1 - a) of its one-hot minus the same share
    assert math.isclose(ga[11] - g0[11], g["label_smoothing"] - share, rel_tol=1e-9)



def test_fused_table_matrix_bytes():
    import bench
    g = _read("ops_nn_fused_table_bytes.txt")
    B, V, s = int(g["B"]), int(g["V"]), int(g["elem_bytes"])
    logits_bytes = bench.logits_bytes(B, V, s)
    assert round(logits_bytes / 1e6) == g["matrix_MB"]
    # one read of the logits + one gradient write + int64 targets
    assert bench.pass_bytes(B, V, s) == 2 * logits_bytes + 8 * B
