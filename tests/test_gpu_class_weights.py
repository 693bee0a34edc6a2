"""Per-class weights (torch F.cross_entropy(weight=...) semantics) on the GPU
against the CPU oracle: per-row losses, the weighted mean, the gradient."""
import numpy as np
import pytest
import torch

import oracle
import vocabulary_cross_entropy_pass_gb300 as pkg
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


# (force_path, tile_kb, stages, weight offset in floats): the planner's
# choice (the stream kernel when rows and weights are 16-byte aligned, 16 KB
# tiles 6 deep), its 32 KB-tile shape, a ring of 4 tiles (too shallow for a
# 16-bit tile and its two weight slots twice: two-stage kernels; enough for
# fp32), a ring of 12 16-KB tiles, the two-stage kernels forced, and weights
# 4 bytes off alignment (two-stage)
ROUTES = [(0, 0, 0, 0), (0, 32, 0, 0), (0, 16, 4, 0), (0, 0, 12, 0), (3, 0, 0, 0),
          (0, 0, 0, 1)]


def expected_path(force, stages, woff, elem_bytes):
    if force == 3 or woff:
        return 3
    if stages and stages < 2 * (1 + 4 // elem_bytes):
        return 3
    return 4


@pytest.mark.parametrize("route", ROUTES, ids=["auto", "tile32", "stages4", "stages12",
                                               "two_stage", "unaligned_w"])
@pytest.mark.parametrize("name", ["c1_bsv4096_f32", "c2_sbv8192_bf16", "c3h_bsv32000_f16_spiked",
                                  "c5_bsv128000_bf16_ls"])
def test_class_weighted_pass(name, route):
    force, tile_kb, stages, woff = route
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(31)
    cw = rng.uniform(0.1, 3.0, w.V).astype(np.float32)
    x = wl.logits(w)
    t = wl.targets(w)
    rngd = np.random.default_rng(32)
    dl = np.array([1.3]) if w.reduce_loss else rngd.uniform(0.5, 2.0, w.N).astype(np.float32)
    ref = oracle.ce(harness.storage_np(x), harness.CODE[w.dtype], w.dim0, w.dim1, w.V,
                    targets=t.numpy().ravel(), label_smoothing=w.label_smoothing,
                    reduce_loss=w.reduce_loss, dloss=dl.astype(np.float64),
                    class_weights=cw.astype(np.float64))
    xd, td = x.to(DEV), t.to(DEV)
    cwd = torch.zeros(w.V + woff, device=DEV)[woff:]
    cwd.copy_(torch.tensor(cw))
    opts = pkg.make_options(force_path=force, tune_tile_kb=tile_kb, tune_stages=stages)
    want = expected_path(force, stages, woff, w.elem_bytes)
    assert pkg.ce_plan_path(xd, opts=pkg.make_options(
        force_path=force, tune_tile_kb=tile_kb, tune_stages=stages,
        class_weights=cwd.data_ptr()))[0] == want
    n = torch.zeros(1, dtype=torch.int64, device=DEV)
    loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=w.label_smoothing, reduce_loss=w.reduce_loss,
                          dloss=torch.tensor(dl, dtype=torch.float32, device=DEV),
                          layout=w.layout, n_non_ignore_out=n, class_weights=cwd, opts=opts)
    assert int(n.item()) == ref["n"]
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, name)
    g = xd.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
    # row scale: dloss over the kept rows' summed target weight (mean), or dloss[r]
    tt = t.numpy().ravel()
    if w.reduce_loss:
        scale = np.full(w.N, dl[0] / cw.astype(np.float64)[tt[tt != -100]].sum())
    else:
        scale = dl.astype(np.float64)
    excess, _ = harness.grad_errors(g, ref["grad"], w.dtype, scale, w.label_smoothing, tt,
                                    weights=cw.astype(np.float64))
    assert excess <= 0.0
    # forward only gives the same losses
    lf = pkg.ce_fwd_only(x.to(DEV), td, label_smoothing=w.label_smoothing,
                         reduce_loss=w.reduce_loss, layout=w.layout, class_weights=cwd,
                         opts=pkg.make_options(force_path=force, tune_tile_kb=tile_kb,
                                               tune_stages=stages))
    harness.check_loss(lf.cpu().numpy(), ref["loss"], w.dtype, name)


def test_unit_weights_equal_unweighted():
    w = wl.WORKLOADS["c2_sbv8192_bf16"]
    x = wl.logits(w).to(DEV)
    t = wl.targets(w).to(DEV)
    a = x.clone()
    la = pkg.ce_fwd_bwd(a, t, label_smoothing=0.1, reduce_loss=True, force_path=3)
    b = x.clone()
    lb = pkg.ce_fwd_bwd(b, t, label_smoothing=0.1, reduce_loss=True,
                        class_weights=torch.ones(w.V, device=DEV))
    harness.check_loss(lb.cpu().numpy(), la.cpu().numpy().astype(np.float64), "bf16")
    tt = t.cpu().numpy().ravel()
    scale = harness.grad_scale(w.N, True, int((tt != -100).sum()))
    excess, _ = harness.grad_errors(b.float().cpu().numpy().astype(np.float64).reshape(w.N, w.V),
                                    a.float().cpu().numpy().astype(np.float64).reshape(w.N, w.V),
                                    "bf16", scale, 0.1, tt)
    assert excess <= 0.0


@pytest.mark.parametrize("force", [1, 2, 5])
def test_weights_refuse_other_paths(force):
    x = torch.zeros(1, 4, 4096, dtype=torch.bfloat16, device=DEV)
    t = torch.zeros(1, 4, dtype=torch.int64, device=DEV)
    with pytest.raises(pkg.CEError):
        pkg.ce_fwd_bwd(x, t, force_path=force, class_weights=torch.ones(4096, device=DEV))


def test_weights_stream_refuses_512_threads():
    x = torch.zeros(1, 4, 4096, dtype=torch.bfloat16, device=DEV)
    t = torch.zeros(1, 4, dtype=torch.int64, device=DEV)
    with pytest.raises(pkg.CEError):
        pkg.ce_fwd_bwd(x, t, class_weights=torch.ones(4096, device=DEV),
                       opts=pkg.make_options(force_path=4, tune_threads=512))
