"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (ctypes handle) and
raises AssertionError when the oracle disagrees with:
  * closed forms (uniform logits give log V for any smoothing; a dominant
    target gives a vanishing loss; rows of the gradient sum to zero);
  * brute force on tiny rows: the unfused softmax -> log -> NLL chain of the
    ops-nn CE fusion article ("Standard approach: three kernels"), written as
    cross-entropy against the smoothed target distribution, in pure Python;
  * central finite differences of that brute-force loss (the gradient);
  * torch.nn.functional.cross_entropy in float64 on the CPU, with autograd
    (a library routine, used only as an independent pin);
  * the vocabulary-parallel combine (hyper-parallel issue #269, section 3.1:
    MAX + SUM all-reduce + target gather over ceil(V/tp) chunks), which must
    equal the unsplit row;
  * exhaustive enumeration of the bf16 / fp16 value sets for rounding.

The functions are plain callables so that tests/test_oracle_mutants.py can run
them against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

F32, BF16, F16 = oracle.F32, oracle.BF16, oracle.F16


def _ce(lib, x32: np.ndarray, t: np.ndarray, a=0.0, reduce=False, dloss=None, ignore=-100):
    """Oracle on a contiguous float32 (N, V) matrix with targets (N,)."""
    N, V = x32.shape
    return oracle.ce(np.ascontiguousarray(x32, dtype=np.float32), F32, 1, N, V,
                     targets=np.asarray(t, dtype=np.int64).reshape(1, N), label_smoothing=a,
                     ignore_idx=ignore, reduce_loss=reduce, dloss=dloss, lib=lib)


def _brute_loss(x, y, a):
    """Cross-entropy of softmax(x) against q = (1-a) onehot(y) + a/V, in
    three explicit steps: softmax, log, weighted negative sum."""
    V = len(x)
    m = max(x)
    e = [math.exp(v - m) for v in x]
    s = math.fsum(e)
    p = [v / s for v in e]
    logp = [math.log(v) for v in p]
    q = [(1.0 - a if j == y else 0.0) + a / V for j in range(V)]
    return -math.fsum(qj * lj for qj, lj in zip(q, logp))


# ---------------------------------------------------------------- closed forms
def pin_uniform_logits_give_log_v(lib):
    for V in (1, 2, 7, 16, 1000, 32000):
        for a in (0.0, 0.1, 0.5, 1.0):
            c = np.float32(3.25)
            x = np.full((3, V), c, dtype=np.float32)
            t = np.array([0, V - 1, V // 2])
            r = _ce(lib, x, t, a=a)
            assert np.allclose(r["loss"], math.log(V), rtol=0, atol=1e-12 * max(1.0, math.log(V))), \
                (V, a, r["loss"])
            assert np.allclose(r["lse"], float(c) + math.log(V), rtol=1e-14)
            # gradient: 1/V - q_j with g = 1
            g = r["grad"]
            for k, y in enumerate(t):
                expect = np.full(V, 1.0 / V - a / V)
                expect[y] -= 1.0 - a
                assert np.allclose(g[k], expect, rtol=1e-12, atol=1e-15), (V, a)


def pin_dominant_target_loss_vanishes(lib):
    V = 50
    x = np.zeros((4, V), dtype=np.float32)
    t = np.array([3, 0, 49, 17])
    for k, y in enumerate(t):
        x[k, y] = 100.0
    r = _ce(lib, x, t)
    assert np.all(r["loss"] < 1e-30) and np.all(r["loss"] >= 0.0), r["loss"]
    for k, y in enumerate(t):
        others = np.delete(r["grad"][k], y)
        assert np.allclose(others, math.exp(-100.0), rtol=1e-9)
        assert abs(r["grad"][k, y]) < 1e-30  # exact: -(V-1) e^-100 ~ -1.8e-42


def pin_single_class_row(lib):
    x = np.array([[5.0], [-3.0]], dtype=np.float32)
    r = _ce(lib, x, np.array([0, 0]), a=0.3)
    assert np.all(r["loss"] == 0.0) and np.all(r["grad"] == 0.0)


def pin_gradient_rows_sum_to_zero(lib):
    rng = np.random.default_rng(5)
    for a in (0.0, 0.1, 0.9):
        x = (rng.standard_normal((6, 333)) * 4).astype(np.float32)
        t = rng.integers(0, 333, 6)
        r = _ce(lib, x, t, a=a, dloss=rng.uniform(0.5, 2.0, 6))
        s = r["grad"].sum(axis=1)
        assert np.all(np.abs(s) < 1e-13), (a, s)


# ---------------------------------------------------------------- brute force
def pin_brute_force_tiny_rows(lib):
    rng = np.random.default_rng(11)
    for V in (1, 2, 3, 5, 8, 16):
        for a in (0.0, 0.1, 0.7):
            x = (rng.standard_normal((V, V)) * 3).astype(np.float32)
            t = np.arange(V)  # every target class once
            r = _ce(lib, x, t, a=a)
            for k in range(V):
                ref = _brute_loss([float(v) for v in x[k]], k, a)
                assert abs(r["loss"][k] - ref) <= 1e-12 * max(1.0, abs(ref)), (V, a, k)


def pin_finite_difference_gradient(lib):
    rng = np.random.default_rng(12)
    h = 1e-5
    for V, a in ((4, 0.0), (9, 0.25), (16, 0.1)):
        x = (rng.standard_normal((2, V)) * 2).astype(np.float32)
        t = np.array([1, V - 1])
        gscale = np.array([1.0, 0.37])
        r = _ce(lib, x, t, a=a, dloss=gscale)
        for k in range(2):
            row = [float(v) for v in x[k]]
            for j in range(V):
                up = row.copy(); up[j] += h
                dn = row.copy(); dn[j] -= h
                fd = (_brute_loss(up, t[k], a) - _brute_loss(dn, t[k], a)) / (2 * h)
                assert abs(r["grad"][k, j] - gscale[k] * fd) < 1e-8, (V, a, k, j)


# ---------------------------------------------------------------- torch float64
def pin_torch_float64_cross_entropy(lib):
    rng = np.random.default_rng(13)
    N, V = 40, 257
    x = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    t = rng.integers(0, V, N)
    t[[3, 17, 18, 39]] = -100
    for a in (0.0, 0.1):
        xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
        tt = torch.tensor(t)
        # per-row losses, per-row upstream gradient
        dl = rng.uniform(0.1, 3.0, N)
        lt = torch.nn.functional.cross_entropy(xt, tt, reduction="none", label_smoothing=a,
                                               ignore_index=-100)
        lt.backward(torch.tensor(dl))
        r = _ce(lib, x, t, a=a, dloss=dl)
        assert np.allclose(r["loss"], lt.detach().numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(r["grad"], xt.grad.numpy(), rtol=1e-10, atol=1e-14)
        # mean over kept rows, upstream gradient of the mean
        xt.grad = None
        lm = torch.nn.functional.cross_entropy(xt, tt, reduction="mean", label_smoothing=a,
                                               ignore_index=-100)
        lm.backward(torch.tensor(1.7, dtype=torch.float64))
        r = _ce(lib, x, t, a=a, reduce=True, dloss=np.array([1.7]))
        assert abs(r["loss"][0] - lm.item()) <= 1e-12 * abs(lm.item())
        assert np.allclose(r["grad"], xt.grad.numpy(), rtol=1e-10, atol=1e-15)
        assert r["n"] == N - 4


# ---------------------------------------------------------------- ignore / count / errors
def pin_ignore_mask_and_count(lib):
    rng = np.random.default_rng(14)
    N, V = 64, 100
    x = rng.standard_normal((N, V)).astype(np.float32)
    t = rng.integers(0, V, N)
    ign = rng.permutation(N)[:9]
    t[ign] = -100
    r = _ce(lib, x, t, a=0.2)
    assert r["n"] == N - 9 and r["err"] == 0
    assert np.all(r["loss"][ign] == 0.0)
    assert np.all(r["grad"][ign] == 0.0)
    keep = np.setdiff1d(np.arange(N), ign)
    assert np.all(r["loss"][keep] > 0.0)
    assert np.all(np.any(r["grad"][keep] != 0.0, axis=1))
    # a non-negative ignore index wins over the range test
    t2 = t.copy(); t2[5] = 7
    r2 = _ce(lib, x, t2, ignore=7)
    assert r2["loss"][5] == 0.0 and np.all(r2["grad"][5] == 0.0)


def pin_out_of_range_target_flags_error(lib):
    x = np.zeros((3, 10), dtype=np.float32)
    r = _ce(lib, x, np.array([2, 10, -5]))
    assert r["err"] & oracle.ERR_TARGET_RANGE
    assert r["loss"][0] == math.log(10) and math.isnan(r["loss"][1]) and math.isnan(r["loss"][2])
    assert np.all(r["grad"][1:] == 0.0) and r["n"] == 3


def pin_all_ignored_mean_is_nan(lib):
    x = np.ones((5, 8), dtype=np.float32)
    r = _ce(lib, x, np.full(5, -100), reduce=True)
    assert math.isnan(r["loss"][0]) and r["n"] == 0 and np.all(r["grad"] == 0.0)


def pin_mean_over_kept_rows(lib):
    rng = np.random.default_rng(15)
    x = rng.standard_normal((10, 30)).astype(np.float32)
    t = rng.integers(0, 30, 10)
    t[[0, 4]] = -100
    per = _ce(lib, x, t)["loss"]
    mean = _ce(lib, x, t, reduce=True)
    assert abs(mean["loss"][0] - math.fsum(per) / 8) < 1e-14
    # reduce: gradient of each kept row is (dloss / n) times its per-row gradient
    g1 = _ce(lib, x, t)["grad"]
    g2 = _ce(lib, x, t, reduce=True, dloss=np.array([2.0]))["grad"]
    assert np.allclose(g2, g1 * 2.0 / 8, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- layout / strides
def pin_layouts_and_strides(lib):
    """(B,SQ,V) and (SQ,B,V) hold the same rows under swapped strides."""
    rng = np.random.default_rng(16)
    B, SQ, V = 3, 5, 40
    x = (rng.standard_normal((B, SQ, V)) * 2).astype(np.float32)
    t = rng.integers(0, V, (B, SQ))
    t[1, 2] = -100
    r_bsv = oracle.ce(x.ravel(), F32, B, SQ, V, strides=(SQ * V, V), targets=t.ravel(),
                      target_strides=(SQ, 1), label_smoothing=0.1, lib=lib)
    xs = np.ascontiguousarray(x.transpose(1, 0, 2))   # (SQ, B, V) storage
    ts = np.ascontiguousarray(t.T)
    r_sbv = oracle.ce(xs.ravel(), F32, SQ, B, V, strides=(B * V, V), targets=ts.ravel(),
                      target_strides=(B, 1), label_smoothing=0.1, lib=lib)
    # row (b, s) of BSV is row (s, b) of SBV
    lb = r_bsv["loss"].reshape(B, SQ)
    ls = r_sbv["loss"].reshape(SQ, B)
    assert np.array_equal(lb, ls.T)
    gb = r_bsv["grad"].reshape(B, SQ, V)
    gs = r_sbv["grad"].reshape(SQ, B, V)
    assert np.array_equal(gb, gs.transpose(1, 0, 2))
    # a strided view of BSV storage read as (SQ,B,V): strides (V, SQ*V)
    r_view = oracle.ce(x.ravel(), F32, SQ, B, V, strides=(V, SQ * V), targets=t.ravel(),
                       target_strides=(1, SQ), label_smoothing=0.1, lib=lib)
    assert np.array_equal(r_view["loss"].reshape(SQ, B), ls)
    # padded rows: row stride larger than V
    pad = np.zeros((B, SQ, V + 8), dtype=np.float32)
    pad[:, :, :V] = x
    r_pad = oracle.ce(pad.ravel(), F32, B, SQ, V, strides=(SQ * (V + 8), V + 8), targets=t.ravel(),
                      target_strides=(SQ, 1), label_smoothing=0.1, lib=lib)
    assert np.array_equal(r_pad["loss"], r_bsv["loss"])


def pin_storage_dtypes_decode(lib):
    """bf16/fp16 storage gives the same result as fp32 storage of the same values."""
    rng = np.random.default_rng(17)
    x = torch.tensor(rng.standard_normal((6, 77)) * 3, dtype=torch.float32)
    t = rng.integers(0, 77, 6)
    for tdt, code in ((torch.bfloat16, BF16), (torch.float16, F16)):
        xs = x.to(tdt)
        bits = xs.view(torch.int16).numpy().view(np.uint16)
        r_bits = oracle.ce(bits, code, 1, 6, 77, targets=t, lib=lib)
        r_f32 = _ce(lib, xs.to(torch.float32).numpy(), t)
        assert np.array_equal(r_bits["loss"], r_f32["loss"])
        assert np.array_equal(r_bits["grad"], r_f32["grad"])


# ---------------------------------------------------------------- split combine
def pin_vocab_split_combine_equals_unsplit(lib):
    rng = np.random.default_rng(18)
    for V, K in ((65536, 8), (128000, 8), (1000, 8), (37, 8), (9, 4)):
        x = rng.standard_normal(V) * 2
        x[rng.integers(0, V)] += 20.0
        y = int(rng.integers(0, V))
        c = -(-V // K)  # ceil(V/K): the last chunk is short (or empty)
        parts = np.stack([oracle.chunk_partials(x, min(k * c, V), min((k + 1) * c, V), y, lib=lib)
                          for k in range(K)])
        lse, xy, S = oracle.combine(parts, lib=lib)
        whole = oracle.chunk_partials(x, 0, V, y, lib=lib)
        lse_whole = whole[0] + math.log(whole[1])
        assert abs(lse - lse_whole) <= 1e-13 * abs(lse_whole), (V, K)
        assert xy == x[y]
        assert abs(S - math.fsum(x)) <= 1e-9 * max(1.0, abs(S))
        # and the unsplit row's lse as reported by the full pass
        r = oracle.ce(x.astype(np.float64).astype(np.float32), F32, 1, 1, V, targets=np.array([y]),
                      want_grad=False, lib=lib)
        x32 = x.astype(np.float32).astype(np.float64)
        parts32 = np.stack([oracle.chunk_partials(x32, min(k * c, V), min((k + 1) * c, V), y, lib=lib)
                            for k in range(K)])
        assert abs(oracle.combine(parts32, lib=lib)[0] - r["lse"][0]) <= 1e-13 * abs(r["lse"][0])


# ---------------------------------------------------------------- rounding
def _all_values(code):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if code == BF16:
        vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    else:
        vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    return np.unique(vals[finite]), bits[finite], vals[finite]


def pin_rounding_is_nearest_even(lib):
    rng = np.random.default_rng(19)
    for code, mant_bits in ((BF16, 7), (F16, 10)):
        table, bits, vals = _all_values(code)
        # exact decode of every finite pattern
        dec = oracle.decode(bits, code, lib=lib)
        assert np.array_equal(dec, vals)
        # random doubles over the whole range: nearest representable value
        probes = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 5, 3000),
                                 rng.uniform(-1e-7, 1e-7, 500)])
        lim = table.max()
        probes = probes[np.abs(probes) < lim]
        got = oracle.round_to(probes, code, lib=lib)
        idx = np.clip(np.searchsorted(table, probes), 1, len(table) - 1)
        lo, hi = table[idx - 1], table[idx]
        best = np.minimum(np.abs(probes - lo), np.abs(probes - hi))
        assert np.all(np.abs(probes - got) == best)
        # exact midpoints between neighbours go to the even significand
        pos = table[(table > 0)]
        mids = (pos[:-1] + pos[1:]) / 2
        sel = rng.choice(len(mids), 2000, replace=False)
        got_m = oracle.round_to(mids[sel], code, lib=lib)
        enc = oracle.encode(mids[sel], code, lib=lib)
        assert np.all((got_m == pos[:-1][sel]) | (got_m == pos[1:][sel]))
        assert np.all((enc & 1) == 0)
        # encode/decode round trip
        assert np.array_equal(oracle.decode(oracle.encode(got, code, lib=lib), code, lib=lib), got)
    # fp32: numpy's float64 -> float32 conversion is correctly rounded
    probes = rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)
    got = oracle.round_to(probes, F32, lib=lib)
    assert np.array_equal(got, probes.astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------- class weights
def _ce_w(lib, x32, t, w, a=0.0, reduce=False, dloss=None):
    N, V = x32.shape
    return oracle.ce(np.ascontiguousarray(x32, dtype=np.float32), F32, 1, N, V,
                     targets=np.asarray(t, dtype=np.int64).reshape(1, N), label_smoothing=a,
                     reduce_loss=reduce, dloss=dloss, class_weights=w, lib=lib)


def _brute_loss_weighted(x, y, a, w):
    """-sum_j q_j w_j log softmax_j, explicit softmax -> log -> weighted sum."""
    V = len(x)
    m = max(x)
    e = [math.exp(v - m) for v in x]
    s = math.fsum(e)
    logp = [math.log(v / s) for v in e]
    q = [(1.0 - a if j == y else 0.0) + a / V for j in range(V)]
    return -math.fsum(qj * wj * lj for qj, wj, lj in zip(q, w, logp))


def pin_class_weights_torch_float64(lib):
    rng = np.random.default_rng(21)
    N, V = 30, 97
    x = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    t = rng.integers(0, V, N)
    t[[2, 11]] = -100
    w = rng.uniform(0.2, 3.0, V)
    for a in (0.0, 0.15):
        xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
        wt = torch.tensor(w)
        tt = torch.tensor(t)
        dl = rng.uniform(0.5, 2.0, N)
        lt = torch.nn.functional.cross_entropy(xt, tt, weight=wt, reduction="none",
                                               label_smoothing=a, ignore_index=-100)
        lt.backward(torch.tensor(dl))
        r = _ce_w(lib, x, t, w, a=a, dloss=dl)
        assert np.allclose(r["loss"], lt.detach().numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(r["grad"], xt.grad.numpy(), rtol=1e-10, atol=1e-14)
        xt.grad = None
        lm = torch.nn.functional.cross_entropy(xt, tt, weight=wt, reduction="mean",
                                               label_smoothing=a, ignore_index=-100)
        lm.backward(torch.tensor(0.8, dtype=torch.float64))
        r = _ce_w(lib, x, t, w, a=a, reduce=True, dloss=np.array([0.8]))
        assert abs(r["loss"][0] - lm.item()) <= 1e-12 * abs(lm.item())
        assert np.allclose(r["grad"], xt.grad.numpy(), rtol=1e-10, atol=1e-15)


def pin_class_weights_brute_force_and_fd(lib):
    rng = np.random.default_rng(22)
    h = 1e-5
    for V, a in ((5, 0.0), (9, 0.3)):
        x = (rng.standard_normal((V, V)) * 2).astype(np.float32)
        w = rng.uniform(0.1, 2.0, V)
        t = np.arange(V)
        r = _ce_w(lib, x, t, w, a=a)
        for k in range(V):
            row = [float(v) for v in x[k]]
            ref = _brute_loss_weighted(row, k, a, w)
            assert abs(r["loss"][k] - ref) <= 1e-12 * max(1.0, abs(ref))
            for j in range(V):
                up = row.copy(); up[j] += h
                dn = row.copy(); dn[j] -= h
                fd = (_brute_loss_weighted(up, k, a, w) - _brute_loss_weighted(dn, k, a, w)) / (2 * h)
                assert abs(r["grad"][k, j] - fd) < 1e-8


def pin_class_weights_closed_forms(lib):
    rng = np.random.default_rng(23)
    V = 64
    w = rng.uniform(0.5, 1.5, V)
    x = np.full((3, V), 1.5, dtype=np.float32)
    t = np.array([0, 17, 63])
    for a in (0.0, 0.2):
        r = _ce_w(lib, x, t, w, a=a)
        # uniform logits: every lse - x_j = log V
        expect = math.log(V) * ((1 - a) * w[t] + a / V * w.sum())
        assert np.allclose(r["loss"], expect, rtol=1e-13)
        # mean divides by the targets' summed weight
        rm = _ce_w(lib, x, t, w, a=a, reduce=True)
        assert abs(rm["loss"][0] - expect.sum() / w[t].sum()) <= 1e-13 * expect.sum()
    # all-ones weights: the unweighted pass
    xr = (rng.standard_normal((4, V)) * 2).astype(np.float32)
    tr = rng.integers(0, V, 4)
    a1 = _ce_w(lib, xr, tr, np.ones(V), a=0.1, reduce=True)
    a0 = _ce(lib, xr, tr, a=0.1, reduce=True)
    assert abs(a1["loss"][0] - a0["loss"][0]) <= 1e-14 * abs(a0["loss"][0])
    assert np.allclose(a1["grad"], a0["grad"], rtol=1e-13, atol=1e-17)


# ---------------------------------------------------------------- lm_head + CE
def pin_linear_ce_identity_weight_is_plain_ce(lib):
    """weight = identity (V = H): the logits are the hidden states themselves."""
    rng = np.random.default_rng(24)
    N, V = 7, 48
    h = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    W = np.eye(V, dtype=np.float32)
    t = rng.integers(0, V, N)
    t[3] = -100
    for a, red in ((0.0, False), (0.2, True)):
        lin = oracle.linear_ce(h, W, F32, N, V, V, t, label_smoothing=a, reduce_loss=red, lib=lib)
        ce = _ce(lib, h, t, a=a, reduce=red)
        assert np.array_equal(lin["loss"], ce["loss"])
        g32 = oracle.round_to(ce["grad"], F32, lib=lib)
        assert np.array_equal(lin["grad_hidden"], g32)
        assert np.array_equal(lin["grad_weight"], g32.T @ h.astype(np.float64))


def pin_linear_ce_torch_float64(lib):
    """The same dataflow in torch float64: logits and the logits gradient
    rounded to float32 where the pass holds float32 tensors."""
    rng = np.random.default_rng(25)
    N, H, V = 9, 24, 61
    h = rng.standard_normal((N, H)).astype(np.float32)
    W = (rng.standard_normal((V, H)) * 0.5).astype(np.float32)
    t = rng.integers(0, V, N)
    t[0] = -100
    for a in (0.0, 0.1):
        h64, W64 = torch.tensor(h, dtype=torch.float64), torch.tensor(W, dtype=torch.float64)
        logits = (h64 @ W64.T).to(torch.float32).to(torch.float64).requires_grad_(True)
        loss = torch.nn.functional.cross_entropy(logits, torch.tensor(t), reduction="mean",
                                                 label_smoothing=a, ignore_index=-100)
        loss.backward(torch.tensor(1.3, dtype=torch.float64))
        dl = logits.grad.to(torch.float32).to(torch.float64)
        r = oracle.linear_ce(h, W, F32, N, H, V, t, label_smoothing=a, reduce_loss=True,
                             dloss=np.array([1.3]), lib=lib)
        assert abs(r["loss"][0] - loss.item()) <= 1e-12 * abs(loss.item())
        assert np.allclose(r["grad_hidden"], (dl @ W64).numpy(), rtol=1e-11, atol=1e-15)
        assert np.allclose(r["grad_weight"], (dl.T @ h64).numpy(), rtol=1e-11, atol=1e-15)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
