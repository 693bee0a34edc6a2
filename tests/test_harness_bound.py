"""The gradient bound of the GPU parity tests (tests/harness.py), checked on
the CPU against the oracle's exact gradients of real workload rows.

Two sides:
  * it is not too tight: an emulation of the pass's float32 arithmetic (the
    rounded logsumexp with a few units of error, exp2 with the error of an
    approximate instruction, the fused multiply-add, then the rounding to the
    storage dtype) passes on every workload family;
  * it bites: gradients with a plausible mistake fail it -- the label
    smoothing share a/V dropped (CSDN "Ascend CANN ops-nn cross-entropy
    fusion", pitfall 3: the smoothing gradient), two 16 KB tiles of a row
    swapped, the exponential off by a factor of two on the elements below
    1e-6, the one-hot term one column off.

Rows are the first rows of each workload (plus its spiked rows), scaled as in
the whole workload (dloss/n of the full batch under reduce_loss)."""
import numpy as np
import pytest

import oracle
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

LOG2E32 = np.float32(1.4426950408889634)


def _rows(name: str, rows: int = 12):
    w = wl.WORKLOADS[name]
    sp, _ = wl.spiked_rows(w)
    pick = np.unique(np.concatenate([np.arange(rows), sp[:2]])).astype(np.int64)
    x = np.concatenate([wl.logits_rows(w, int(r), int(r) + 1) .float().numpy() for r in pick])
    xs = np.concatenate([harness.storage_np(wl.logits_rows(w, int(r), int(r) + 1)) for r in pick])
    t = wl.targets(w).reshape(-1).numpy()[pick]
    n_full = w.N - int(np.floor(w.ignore_frac * w.N))
    g = np.full(len(pick), 1.0 / n_full) if w.reduce_loss else np.ones(len(pick))
    sub = w.with_(dim0=1, dim1=len(pick), reduce_loss=False)
    ref = oracle.ce(xs, harness.CODE[w.dtype], 1, len(pick), w.V, targets=t,
                    label_smoothing=w.label_smoothing, dloss=g)
    return w, sub, x.astype(np.float32), t, g, ref


def _emulate_f32(x32, t, g, a, lse, dtype, rng):
    """The pass's gradient in float32 as the kernels compute it, with errors
    of the size the hardware makes: lse off by up to two float32 units, each
    exp2 off by up to 2^-22 relative; then rounded to the storage dtype."""
    N, V = x32.shape
    lse32 = (lse * (1 + rng.uniform(-2, 2, N) * 2.0 ** -24)).astype(np.float32)
    nll = (-lse32 * LOG2E32).astype(np.float32)
    arg = (x32.astype(np.float64) * np.float64(LOG2E32) + nll[:, None]).astype(np.float32)
    e = np.exp2(arg.astype(np.float64)) * (1 + rng.uniform(-1, 1, arg.shape) * 2.0 ** -22)
    e = e.astype(np.float32)
    a_over_v = np.float32(a / V)
    G = g.astype(np.float32)[:, None]
    bb = (G * a_over_v).astype(np.float32)
    o = (e.astype(np.float64) * G + (-bb)).astype(np.float32).astype(np.float64)
    keep = t != -100
    rows = np.nonzero(keep)[0]
    ey = e[rows, t[rows]].astype(np.float64)
    oy = (ey * G[rows, 0] - bb[rows, 0]).astype(np.float32)
    o[rows, t[rows]] = (oy - (G[rows, 0] * np.float32(1 - a)).astype(np.float32)).astype(np.float32)
    o[~keep] = 0.0
    return oracle.round_to(o, harness.CODE[dtype]) if dtype != "f32" else o


FAMILIES = ["c1_bsv4096_f32", "c2_sbv8192_bf16", "c3_bsv32000_bf16_spiked",
            "c3h_bsv32000_f16_spiked", "c4_bsv65536_bf16_split8", "c5_bsv128000_bf16",
            "c5_bsv128000_bf16_ls", "c5_bsv128000_f32_ls"]


@pytest.mark.parametrize("name", FAMILIES)
def test_bound_admits_float32_arithmetic(name):
    w, sub, x32, t, g, ref = _rows(name)
    rng = np.random.default_rng(7)
    for _ in range(3):
        got = _emulate_f32(x32, t, g, w.label_smoothing, ref["lse"], w.dtype, rng)
        excess, _ = harness.grad_errors(got, ref["grad"], w.dtype, g, w.label_smoothing, t)
        assert excess <= 0.0, f"{name}: a float32 pass exceeds the bound by {excess:.3e}"


def _fails(w, ref, g, t, wrong):
    got = wrong if w.dtype == "f32" else oracle.round_to(wrong, harness.CODE[w.dtype])
    excess, _ = harness.grad_errors(got, ref["grad"], w.dtype, g, w.label_smoothing, t)
    return excess > 0.0


@pytest.mark.parametrize("name", ["c5_bsv128000_bf16_ls", "c5_bsv128000_f32_ls",
                                  "c4_bsv65536_bf16_split8", "c2_sbv8192_bf16"])
def test_bound_rejects_dropped_smoothing_share(name):
    w, sub, x32, t, g, ref = _rows(name)
    keep = t != -100
    wrong = ref["grad"].copy()
    wrong[keep] += (g[keep] * w.label_smoothing / w.V)[:, None]
    assert _fails(w, ref, g, t, wrong)


@pytest.mark.parametrize("name", ["c5_bsv128000_bf16_ls", "c5_bsv128000_f32_ls",
                                  "c3h_bsv32000_f16_spiked", "c1_bsv4096_f32"])
def test_bound_rejects_swapped_tiles(name):
    w, sub, x32, t, g, ref = _rows(name)
    tile = 16384 // w.elem_bytes
    if w.V < 2 * tile:
        tile = w.V // 4
    wrong = ref["grad"].copy()
    wrong[:, :tile], wrong[:, tile:2 * tile] = ref["grad"][:, tile:2 * tile], ref["grad"][:, :tile]
    assert _fails(w, ref, g, t, wrong)


@pytest.mark.parametrize("name", ["c5_bsv128000_bf16_ls", "c5_bsv128000_bf16",
                                  "c5_bsv128000_f32_ls", "c2_sbv8192_bf16"])
def test_bound_rejects_exponential_off_by_two_below_1e6(name):
    w, sub, x32, t, g, ref = _rows(name)
    keep = t != -100
    # softmax from the exact gradient: p = grad/g + q
    p = ref["grad"][keep] / g[keep, None] + w.label_smoothing / w.V
    rows = np.nonzero(keep)[0]
    p[np.arange(len(rows)), t[rows]] += 1 - w.label_smoothing
    small = np.abs(ref["grad"][keep]) < 1e-6
    wrong = ref["grad"].copy()
    wrong[keep] = np.where(small, ref["grad"][keep] + g[keep, None] * p, ref["grad"][keep])
    assert _fails(w, ref, g, t, wrong)


@pytest.mark.parametrize("name", ["c5_bsv128000_bf16_ls", "c3_bsv32000_bf16_spiked"])
def test_bound_rejects_one_hot_in_the_wrong_column(name):
    w, sub, x32, t, g, ref = _rows(name)
    keep = np.nonzero(t != -100)[0]
    wrong = ref["grad"].copy()
    y = t[keep]
    y2 = (y + 1) % w.V
    d = g[keep] * (1 - w.label_smoothing)
    wrong[keep, y] += d
    wrong[keep, y2] -= d
    assert _fails(w, ref, g, t, wrong)


def test_exact_rounding_passes_and_zero_rows_are_exact():
    w, sub, x32, t, g, ref = _rows("c5_bsv128000_bf16_ls")
    r = oracle.round_to(ref["grad"], oracle.BF16)
    excess, _ = harness.grad_errors(r, ref["grad"], "bf16", g, w.label_smoothing, t)
    assert excess <= 0.0
    # an ignored row must be exactly zero: a tiny nonzero value fails
    ign = np.nonzero(t == -100)[0]
    if len(ign):
        wrong = r.copy()
        wrong[ign[0], 0] = 1e-30
        excess, _ = harness.grad_errors(wrong, ref["grad"], "bf16", g, w.label_smoothing, t)
        assert excess > 0.0
