"""Shared helpers of the GPU parity tests: run a workload through the C ABI
(via the ctypes binding) and through the CPU oracle on the same input bytes,
and compare element by element with the stated tolerances.

Tolerances (per token row; from the precision contract of the pass):
  loss  : |loss - ref| <= tol * max(|ref|, 1), tol = 1e-5 for fp32 logits,
          2e-3 for bf16/fp16 logits (the max(.,1) guards rows whose loss is
          near zero, where a relative error says nothing);
  grad  : fp32: |g - ref| <= 1e-6;  bf16/fp16: |g - round(ref)| <= ulp(ref) + 1e-6,
          ulp() the spacing of the storage format at |ref| (its subnormal
          spacing below the smallest normal);
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
    p, emin = (8, -126) if dtype == "bf16" else (11, -14)
    e = np.frexp(np.abs(ref))[1] - 1          # exponent of the leading bit
    e = np.maximum(e, emin)
    return np.ldexp(1.0, e - (p - 1))


def grad_errors(g: np.ndarray, ref: np.ndarray, dtype: str) -> tuple[float, np.ndarray]:
    """Max excess over tolerance (<= 0 passes) and the per-element bound."""
    if dtype == "f32":
        bound = np.full(ref.shape, 1e-6)
        err = np.abs(g - ref)
    else:
        r = oracle.round_to(ref, CODE[dtype])
        bound = ulp(r, dtype) + 1e-6
        err = np.abs(g - r)
    return float(np.max(err - bound)) if err.size else 0.0, err


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
    excess, err_abs = grad_errors(g, ref["grad"], w.dtype)
    out["grad_abs_max"] = float(err_abs.max())
    assert excess <= 0.0, f"{w.name}: gradient exceeds tolerance by {excess:.3e}"
    return out
