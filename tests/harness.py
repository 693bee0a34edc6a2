"""Shared helpers of the GPU parity tests: run a workload through the C ABI
(via the ctypes binding) and through the CPU oracle on the same input bytes,
and compare element by element with the stated tolerances.

Tolerances (per token row; from the precision contract of the pass):
  loss  : |loss - ref| <= tol * max(|ref|, 1), tol = 1e-5 for fp32 logits,
          2e-3 for bf16/fp16 logits (the max(.,1) guards rows whose loss is
          near zero, where a relative error says nothing);
  grad  : the contract's absolute 1e-6 is read as stated for a unit upstream
          gradient: every element of row r is the row's scale g_r = dloss/n
          (reduce_loss) or dloss[r] times a difference of terms of order one,
          g_r (p_j - q_j) with p the softmax and q the smoothed one-hot target
          (times the class weights in the weighted pass).  The bound is
            bf16/fp16: |g - ref| <= ulp(ref) + |g_r| min(1e-6, 4e-6 M_j)
            fp32:      |g - ref| <=          |g_r| min(1e-6, 8e-6 M_j)
          with M_j = |ref_j|/|g_r| + 2|q_j| >= p_j + |q_j|, the size of the
          terms whose difference the element is (the float32 arithmetic of
          the pass errs by a few 1e-6 of them: the exponential, the rounded
          logsumexp, the final fused multiply-add).  ulp() is the spacing of
          the storage format at the exact |ref| (its subnormal spacing below
          the smallest normal), the distance taken from the exact reference.
          It is never looser than the contract's floor scaled by g_r, and at
          the (1, 512, 128000) bf16 workload with smoothing (g_r = 1/461) it
          resolves the smoothing share g_r a/V = 1.7e-9 that a plain 1e-6
          floor -- or 1e-6 g_r -- would hide;
  mask  : ignored rows have loss exactly 0 and a gradient of exact zeros;
  count : n_non_ignore exactly equal.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

CODE = {"f32": oracle.F32, "bf16": oracle.BF16, "f16": oracle.F16}
LOSS_TOL = {"f32": 1e-5, "bf16": 2e-3, "f16": 2e-3}


def storage_np(x: torch.Tensor) -> np.ndarray:
    """Raw storage of a CPU tensor as numpy (float32, or uint16 bit patterns)."""
    x = x.contiguous()
    if x.dtype == torch.float32:
        return x.numpy().ravel()
    return x.view(torch.int16).numpy().view(np.uint16).ravel()


def ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the storage format (bf16 or fp16) at |ref|; its smallest
    (subnormal) spacing at and below the smallest normal, and at zero."""
    p, emin = (8, -126) if dtype == "bf16" else (11, -14)
    a = np.abs(ref)
    e = np.frexp(a)[1] - 1          # exponent of the leading bit
    e = np.where(a == 0, emin, np.maximum(e, emin))
    return np.ldexp(1.0, e - (p - 1))


def grad_scale(N: int, reduce_loss: bool, n: int, dloss=None) -> np.ndarray:
    """|g_r| of every flattened row: dloss/n (or 1/n) under reduce_loss, else
    dloss[r] (or 1).  With every row ignored (n = 0) the scale is 0: the
    gradient must then be exactly zero."""
    if reduce_loss:
        d = 1.0 if dloss is None else float(np.ravel(dloss)[0])
        return np.full(N, abs(d) / n if n > 0 else 0.0)
    if dloss is None:
        return np.ones(N)
    return np.abs(np.asarray(dloss, dtype=np.float64).ravel())


KAPPA = {"f32": 8e-6, "bf16": 4e-6, "f16": 4e-6}


def grad_bound(ref: np.ndarray, dtype: str, scale, label_smoothing: float, targets,
               ignore_idx: int = -100, weights=None) -> np.ndarray:
    """Per-element bound of |g - ref| (see the module docstring).

    ref: (N, V) exact gradient; scale: |g_r| per row, (N,) or one value;
    targets: (N,) flattened row targets; weights: (V,) class weights or None."""
    N, V = ref.shape
    s = np.broadcast_to(np.abs(np.asarray(scale, dtype=np.float64)).reshape(-1), (N,))[:, None]
    a = float(label_smoothing)
    w = np.ones(V) if weights is None else np.abs(np.asarray(weights, dtype=np.float64))
    safe = np.where(s > 0, s, 1.0)
    y = np.asarray(targets, dtype=np.int64).reshape(-1)
    kept = (y != ignore_idx) & (y >= 0) & (y < V)
    # ignored and out-of-range rows are exact zeros: no term, no floor
    M = np.abs(ref) / safe + np.where(kept[:, None], (2.0 * a / V) * w[None, :], 0.0)
    rows = np.nonzero(kept)[0]
    M[rows, y[rows]] += 2.0 * (1.0 - a) * w[y[rows]]
    floor = s * np.minimum(1e-6, KAPPA[dtype] * M)
    return floor if dtype == "f32" else ulp(ref, dtype) + floor


def grad_errors(g: np.ndarray, ref: np.ndarray, dtype: str, scale, label_smoothing: float,
                targets, ignore_idx: int = -100, weights=None) -> tuple[float, np.ndarray]:
    """Max excess over the bound (<= 0 passes) and the per-element error.

    g, ref: (N, V) gradients (ref exact, double); the other arguments as for
    grad_bound."""
    g = np.asarray(g, dtype=np.float64).reshape(ref.shape)
    err = np.abs(g - ref)
    if not err.size:
        return 0.0, err
    bound = grad_bound(ref, dtype, scale, label_smoothing, targets, ignore_idx, weights)
    return float(np.max(err - bound)), err


def check_grad(g, ref: dict, w: wl.Workload, t, dloss=None, weights=None, what="") -> float:
    """Assert the gradient of workload w (targets t, oracle result ref with
    the same dloss) within grad_bound; returns the largest error."""
    scale = grad_scale(w.N, w.reduce_loss, ref["n"], dloss)
    tt = t.contiguous().numpy().ravel() if isinstance(t, torch.Tensor) else np.ravel(t)
    excess, err = grad_errors(np.asarray(g, dtype=np.float64).reshape(w.N, w.V), ref["grad"],
                              w.dtype, scale, w.label_smoothing, tt, w.ignore_idx, weights)
    assert excess <= 0.0, f"{what or w.name}: gradient exceeds tolerance by {excess:.3e}"
    return float(err.max(initial=0.0))


def oracle_run(w: wl.Workload, x_cpu: torch.Tensor, t_cpu: torch.Tensor, dloss=None,
               want_grad=True, strides=None, target_strides=None):
    return oracle.ce(storage_np(x_cpu), CODE[w.dtype], w.dim0, w.dim1, w.V, strides=strides,
                     targets=t_cpu.contiguous().numpy().ravel(), target_strides=target_strides,
                     label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                     reduce_loss=w.reduce_loss,
                     dloss=None if dloss is None else np.asarray(dloss, dtype=np.float64),
                     want_grad=want_grad)


def check_loss(got: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    got = np.asarray(got, dtype=np.float64)
    tol = LOSS_TOL[dtype]
    both_nan = np.isnan(got) & np.isnan(ref)
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)
    rel[both_nan] = 0.0
    assert not np.any(np.isnan(rel)), f"{what}: NaN mismatch"
    assert rel.max(initial=0.0) <= tol, f"{what}: loss rel err {rel.max():.3e} > {tol}"
    return float(rel.max(initial=0.0))


def run_gpu_vs_oracle(w: wl.Workload, force_path: int = 0, num_vocab_chunks: int | None = None,
                      per_row_dloss: bool = False):
    """Full parity of one workload; returns a dict of the worst errors."""
    import vocabulary_cross_entropy_pass_gb300 as pkg
    dev = torch.device("cuda")
    x = wl.logits(w)
    t = wl.targets(w)
    K = w.vocab_chunks if num_vocab_chunks is None else num_vocab_chunks
    dl_np = None
    dl = None
    if w.reduce_loss:
        dl_np = np.array([1.0])
    elif per_row_dloss:
        rng = np.random.default_rng(w.seed + 99)
        dl_np = rng.uniform(0.25, 2.0, w.N).astype(np.float32).astype(np.float64)
        dl = torch.tensor(dl_np, dtype=torch.float32, device=dev)
    ref = oracle_run(w, x, t, dloss=dl_np)

    xd = x.to(dev)
    td = t.to(dev)
    n = torch.zeros(1, dtype=torch.int64, device=dev)
    ws = torch.empty(pkg.ce_workspace_bytes(w.dim0, w.dim1, w.V, xd.dtype,
                                            pkg.make_options(force_path, K)),
                     dtype=torch.uint8, device=dev)
    loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                          reduce_loss=w.reduce_loss, dloss=dl, layout=w.layout,
                          n_non_ignore_out=n, workspace=ws, force_path=force_path,
                          num_vocab_chunks=K)
    st, err = pkg.ce_get_error(ws)
    assert st == 0 and err == 0, (st, err)
    assert int(n.item()) == ref["n"]

    out = {}
    out["loss_rel"] = check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, w.name)
    g = xd.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
    ign = wl.ignored_rows(w)
    assert np.all(g[ign] == 0.0), "ignored rows must have an exactly zero gradient"
    if not w.reduce_loss:
        assert np.all(loss.cpu().numpy()[ign] == 0.0)
    out["grad_abs_max"] = check_grad(g, ref, w, t, dloss=dl_np)
    return out
