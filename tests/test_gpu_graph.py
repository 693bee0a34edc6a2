"""The pass inside a CUDA graph (TENPU #29 section 7 lists is_cg_capturable;
this library allocates nothing and never synchronises inside a call, so the
whole pass -- count kernel, main kernel, mean -- can be captured once and
replayed on new inputs copied into the same buffers)."""
import numpy as np
import pytest
import torch

import vocabulary_cross_entropy_pass_gb300 as pkg
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("name,path", [("c5_bsv128000_bf16_ls", 0), ("c2_sbv8192_bf16", 0),
                                       ("c3_bsv32000_bf16_spiked", 2), ("c4_bsv65536_bf16_split8", 3)])
def test_graph_capture_and_replay(name, path):
    w = wl.WORKLOADS[name]
    x_a = wl.logits(w)
    t = wl.targets(w)
    x_b = wl.logits(w.with_(seed=w.seed + 77))
    xs = x_a.to(DEV)                     # static input buffer of the graph
    ts = t.to(DEV)
    loss = torch.empty(1 if w.reduce_loss else w.N, dtype=torch.float32, device=DEV)
    opts = pkg.make_options(force_path=path, num_vocab_chunks=w.vocab_chunks if path in (2, 3) else 0)
    ws = torch.empty(pkg.ce_workspace_bytes(w.dim0, w.dim1, w.V, xs.dtype, opts), dtype=torch.uint8,
                     device=DEV)
    kw = dict(label_smoothing=w.label_smoothing, reduce_loss=w.reduce_loss, layout=w.layout,
              loss_out=loss, workspace=ws, opts=opts)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):        # warm-up outside the capture
        pkg.ce_fwd_bwd(xs, ts, **kw)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    xs.copy_(x_a.to(DEV))
    with torch.cuda.graph(g):
        pkg.ce_fwd_bwd(xs, ts, **kw)
    for x_in in (x_a, x_b, x_a):
        xs.copy_(x_in.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        dl = np.array([1.0]) if w.reduce_loss else None
        ref = harness.oracle_run(w, x_in, t, dloss=dl)
        harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, name)
        gr = xs.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
        harness.check_grad(gr, ref, w, t, dloss=dl)
