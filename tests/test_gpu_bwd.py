"""The separate backward (ce_bwd from a saved lse) and the autograd wrapper,
against the CPU oracle: ce_fwd_only saves lse and the kept-row count, ce_bwd
writes the gradient for an upstream gradient known only afterwards."""
import numpy as np
import pytest
import torch

import vocabulary_cross_entropy_pass_gb300 as pkg
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _upstream(w, rng):
    if w.reduce_loss:
        return np.array([1.7])
    return rng.uniform(0.25, 2.0, w.N).astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("name", ["c1_bsv4096_f32", "c2_sbv8192_bf16", "c3h_bsv32000_f16_spiked",
                                  "c5_bsv128000_bf16_ls"])
@pytest.mark.parametrize("inplace", [False, True])
def test_fwd_only_then_bwd(name, inplace):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(3)
    x = wl.logits(w)
    t = wl.targets(w)
    dl = _upstream(w, rng)
    ref = harness.oracle_run(w, x, t, dloss=dl)
    xd, td = x.to(DEV), t.to(DEV)
    lse = torch.empty(w.N, dtype=torch.float32, device=DEV)
    n = torch.empty(1, dtype=torch.int64, device=DEV)
    loss = pkg.ce_fwd_only(xd, td, label_smoothing=w.label_smoothing, reduce_loss=w.reduce_loss,
                           layout=w.layout, lse_out=lse, n_non_ignore_out=n)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, name)
    g = pkg.ce_bwd(xd, td, lse, label_smoothing=w.label_smoothing, reduce_loss=w.reduce_loss,
                   dloss=torch.tensor(dl, dtype=torch.float32, device=DEV), n_non_ignore=n,
                   grad=xd if inplace else None, layout=w.layout)
    if inplace:
        assert g.data_ptr() == xd.data_ptr()
    else:
        assert torch.equal(xd.cpu(), x)  # logits untouched
    gn = g.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
    harness.check_grad(gn, ref, w, t, dloss=dl)


@pytest.mark.parametrize("V,dtype", [(4095, "bf16"), (7, "f32"), (1000, "f16")])
def test_bwd_unaligned_rows(V, dtype):
    w = wl.Workload("u", 1, 9, V, dtype, sigma=2.0, ignore_frac=0.2, label_smoothing=0.2, seed=V)
    x = wl.logits(w)
    t = wl.targets(w)
    ref = harness.oracle_run(w, x, t)
    xd, td = x.to(DEV), t.to(DEV)
    lse = torch.empty(w.N, dtype=torch.float32, device=DEV)
    pkg.ce_fwd_only(xd, td, label_smoothing=0.2, lse_out=lse)
    g = pkg.ce_bwd(xd, td, lse, label_smoothing=0.2)
    harness.check_grad(g.float().cpu().numpy(), ref, w, t)


@pytest.mark.parametrize("name", ["c2_sbv8192_bf16", "c3_bsv32000_bf16_spiked", "c1_bsv4096_f32"])
@pytest.mark.parametrize("inplace", [False, True])
def test_autograd_wrapper(name, inplace):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(4)
    x = wl.logits(w)
    t = wl.targets(w)
    dl = _upstream(w, rng)
    ref = harness.oracle_run(w, x, t, dloss=dl)
    xd = x.to(DEV).requires_grad_(True)
    loss = pkg.parallel_cross_entropy(xd, t.to(DEV), label_smoothing=w.label_smoothing,
                                      reduce_loss=w.reduce_loss, layout=w.layout,
                                      inplace_grad=inplace)
    assert loss.shape == (() if w.reduce_loss else t.shape)
    harness.check_loss(loss.detach().cpu().numpy().reshape(-1), ref["loss"], w.dtype, name)
    gout = torch.tensor(dl.reshape(loss.shape) if not w.reduce_loss else dl[0],
                        dtype=torch.float32, device=DEV)
    loss.backward(gout)
    gn = xd.grad.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
    harness.check_grad(gn, ref, w, t, dloss=dl)


def test_fused_and_split_backward_agree():
    w = wl.WORKLOADS["c5_bsv128000_bf16_ls"]
    x = wl.logits(w).to(DEV)
    t = wl.targets(w).to(DEV)
    a = x.clone()
    pkg.ce_fwd_bwd(a, t, label_smoothing=0.1, reduce_loss=True)
    lse = torch.empty(w.N, dtype=torch.float32, device=DEV)
    n = torch.empty(1, dtype=torch.int64, device=DEV)
    pkg.ce_fwd_only(x, t, label_smoothing=0.1, reduce_loss=True, lse_out=lse, n_non_ignore_out=n)
    b = pkg.ce_bwd(x, t, lse, label_smoothing=0.1, reduce_loss=True, n_non_ignore=n)
    ga = a.float().cpu().numpy().astype(np.float64).reshape(w.N, w.V)
    gb = b.float().cpu().numpy().astype(np.float64).reshape(w.N, w.V)
    scale = harness.grad_scale(w.N, True, int(n.item()))
    excess, _ = harness.grad_errors(gb, ga, "bf16", scale, 0.1, t.cpu().numpy().ravel())
    assert excess <= 0.0


def test_dist_process_group_is_refused():
    x = torch.zeros(1, 2, 8, device=DEV)
    t = torch.zeros(1, 2, dtype=torch.int64, device=DEV)
    with pytest.raises(NotImplementedError):
        pkg.parallel_cross_entropy(x, t, dist_process_group=object())


@pytest.mark.parametrize("V,dtype,gshift", [(20011, "bf16", 0), (20011, "bf16", 1), (8193, "f16", 0),
                                            (10007, "f32", 0), (10007, "f32", 3)])
def test_bwd_unaligned_rows_wide(V, dtype, gshift):
    """Rows off the 16-byte grid over several 16 KB chunks: with the gradient
    at the logits' offset from a 16-byte boundary (gshift 0) the chunks move
    in 16-byte vectors between a scalar head and tail; a gradient view
    shifted by gshift elements takes the element-by-element kernel.  The
    gradient buffer's padding stays untouched."""
    w = wl.Workload("uw", 1, 13, V, dtype, sigma=2.0, ignore_frac=0.2, label_smoothing=0.1, seed=V + gshift)
    x = wl.logits(w)
    t = wl.targets(w)
    ref = harness.oracle_run(w, x, t)
    xd, td = x.to(DEV), t.to(DEV)
    lse = torch.empty(w.N, dtype=torch.float32, device=DEV)
    pkg.ce_fwd_only(xd, td, label_smoothing=0.1, lse_out=lse)
    gbuf = torch.zeros(1, 13, V + 8, dtype=xd.dtype, device=DEV)
    gview = gbuf[:, :, gshift:gshift + V]
    g = pkg.ce_bwd(xd, td, lse, label_smoothing=0.1, grad=gview)
    harness.check_grad(g.float().cpu().numpy(), ref, w, t)
    host = gbuf.cpu()
    assert torch.all(host[:, :, :gshift] == 0) and torch.all(host[:, :, gshift + V:] == 0)
    assert torch.equal(xd.cpu(), x)
