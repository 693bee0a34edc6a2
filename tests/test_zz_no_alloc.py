"""ce_fwd_bwd_noalloc: the pass for callers that must not allocate device
memory per call (runtimes that plan all device memory before they start and
give custom operators no workspace; latency-critical loops that cannot risk
cudaMalloc's device synchronisation or failure).  Its scratch is the library's
own fixed device array, so these tests compare it with ce_fwd_bwd, which uses a
caller-provided workspace, on the same inputs, bit for bit, twice in a row
with new inputs for the second call (which reuses the array the first one
left behind).

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from vocabulary_cross_entropy_pass_gb300 import _lib
from vocabulary_cross_entropy_pass_gb300 import workloads as wl


def _noalloc_c(x, t, loss, a, reduce, opts=None):
    """Call the C entry point directly through ctypes."""
    lib = _lib.load()
    d0, d1, V = x.shape
    st = _lib.i64_array(x.stride())
    ts = _lib.i64_array(t.stride())
    stream = torch.cuda.current_stream().cuda_stream if x.is_cuda else 0
    return lib.ce_fwd_bwd_noalloc(ctypes.c_void_p(x.data_ptr()), {torch.float32: 0,
                                  torch.bfloat16: 1, torch.float16: 2}[x.dtype], 0, d0, d1, V, st,
                                  ctypes.c_void_p(t.data_ptr()), ts, float(a), -100, int(reduce),
                                  None, ctypes.c_void_p(loss.data_ptr()),
                                  ctypes.c_void_p(x.data_ptr()), None,
                                  ctypes.byref(opts) if opts is not None else None,
                                  ctypes.c_void_p(stream))


def test_oversized_problems_are_rejected_on_the_host():
    # no GPU needed: the size test runs before any CUDA call
    from vocabulary_cross_entropy_pass_gb300 import build
    build.build()
    lib = _lib.load()
    loss = ctypes.c_void_p(0x3000)

    def call(d1, V, **o):
        opts = _lib.make_options(**o)
        return lib.ce_fwd_bwd_noalloc(ctypes.c_void_p(0x1000), 1, 0, 1, d1, V,
                                      _lib.i64_array((d1 * V, V, 1)), ctypes.c_void_p(0x2000),
                                      _lib.i64_array((d1, 1)), 0.0, -100, 1, None, loss,
                                      ctypes.c_void_p(0x1000), None, ctypes.byref(opts), None)
    assert call(600_000, 4096) == 4                 # per-row losses alone exceed 2 MiB
    assert call(20_000, 128000, force_path=3) == 4  # two-stage partials exceed 2 MiB
    assert call(8, 4096, tune_threads=300) == 1     # ordinary argument checks still apply


# (workload, forced path, vocabulary chunks): the warp path, the stream path
# with its in-kernel mean and row counter in the scratch header, the stream
# path split into 8 chunks (its chunk partials in the scratch), the two-stage
# path with its partials in the scratch, fp32 rows, and rows off the 16-byte
# grid (odd width: the stream kernel with scalar edges, and the plain-load
# kernel forced)
CASES = [("c2_sbv8192_bf16", 0, 0), ("c5_bsv128000_bf16_ls", 0, 0),
         ("c4_bsv65536_bf16_split8", 0, 8), ("c3_bsv32000_bf16_spiked", 3, 0),
         ("c1_bsv4096_f32", 0, 0), ("odd_50257_bf16", 0, 0), ("odd_50257_bf16", 6, 0)]
ODD = wl.Workload("odd_50257_bf16", 1, 64, 50257, "bf16", sigma=2.0, ignore_frac=0.1,
                  label_smoothing=0.1, reduce_loss=True, seed=5257)


@pytest.mark.gpu
@pytest.mark.parametrize("name,path,chunks", CASES)
def test_noalloc_matches_workspace_entry_point(name, path, chunks):
    """Same plan, same kernels: the results must equal ce_fwd_bwd's bit for
    bit.  The second call gets other logits and targets, so scratch the first
    call left behind (row counter, ticket, partials) cannot pass for the
    second call's own."""
    import vocabulary_cross_entropy_pass_gb300 as pkg
    w0 = ODD if name == ODD.name else wl.WORKLOADS[name]
    dev = torch.device("cuda")
    opts = _lib.make_options(force_path=path, num_vocab_chunks=chunks)
    for call in range(2):   # two calls in a row share the fixed scratch
        w = w0.with_(seed=w0.seed + 101 * call)
        x = wl.logits(w).to(dev)
        t = wl.targets(w).to(dev)
        if call:
            t = t.roll(1)     # ignored rows move too
        xa, xb = x.clone(), x.clone()
        la = pkg.ce_fwd_bwd(xa, t, label_smoothing=w.label_smoothing,
                            reduce_loss=w.reduce_loss, force_path=path, num_vocab_chunks=chunks)
        lb = torch.full_like(la, float("nan"))
        rc = _noalloc_c(xb, t, lb, w.label_smoothing, w.reduce_loss, opts)
        assert rc == 0, _lib.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert torch.equal(la, lb), f"{name} call {call}: losses differ"
        assert torch.equal(xa, xb), f"{name} call {call}: gradients differ"
        assert not torch.equal(xb, x)  # the gradient was written


@pytest.mark.gpu
def test_noalloc_python_binding():
    import vocabulary_cross_entropy_pass_gb300 as pkg
    w = wl.WORKLOADS["c2_sbv8192_bf16"]
    dev = torch.device("cuda")
    x = wl.logits(w).to(dev)
    t = wl.targets(w).to(dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    xa = x.clone()
    ref = pkg.ce_fwd_bwd(xa, t, label_smoothing=w.label_smoothing, reduce_loss=True)
    pkg.ce_fwd_bwd_noalloc(x, t, loss, label_smoothing=w.label_smoothing, reduce_loss=True)
    assert torch.equal(loss, ref) and torch.equal(x, xa)


@pytest.mark.gpu
def test_noalloc_error_word():
    """Out-of-range targets set the error word of the library's own scratch,
    which ce_noalloc_get_error reads; the next clean pass clears it."""
    import vocabulary_cross_entropy_pass_gb300 as pkg
    w = wl.Workload("oor_noalloc", 1, 6, 8192, "bf16", sigma=2.0, ignore_frac=0.0, seed=73)
    dev = torch.device("cuda")
    t = wl.targets(w)
    t[0, 2] = 8192
    t[0, 4] = -7
    x = wl.logits(w).to(dev)
    loss = torch.empty(6, dtype=torch.float32, device=dev)
    pkg.ce_fwd_bwd_noalloc(x, t.to(dev), loss, reduce_loss=False)
    st, err = pkg.ce_noalloc_get_error()
    assert err & 1 and st == 6
    lc = loss.cpu()
    assert torch.isnan(lc[2]) and torch.isnan(lc[4]) and torch.isfinite(lc[[0, 1, 3, 5]]).all()
    pkg.ce_fwd_bwd_noalloc(wl.logits(w).to(dev), wl.targets(w).to(dev), loss, reduce_loss=False)
    assert pkg.ce_noalloc_get_error() == (0, 0)
