"""Edge cases of the GPU pass against the CPU oracle: tiny and unaligned
vocabularies, padded and transposed rows, empty and ragged vocabulary chunks,
all-ignored rows, out-of-range targets, N = 0, forward-only, determinism of
the mean, and the full-size throughput workload on sampled rows."""
import math

import numpy as np
import pytest
import torch

import oracle
import vocabulary_cross_entropy_pass_gb300 as pkg
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _compare(w, x_cpu, t_cpu, loss, g_dev, n_dev=None, strides=None, tstrides=None):
    """Oracle on the CPU copy (same storage/strides) vs GPU outputs."""
    dl = np.array([1.0]) if w.reduce_loss else None
    ref = oracle.ce(harness.storage_np(x_cpu), harness.CODE[w.dtype], w.dim0, w.dim1, w.V,
                    strides=strides, targets=t_cpu.contiguous().numpy().ravel(),
                    target_strides=tstrides,
                    label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                    reduce_loss=w.reduce_loss, dloss=dl)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, w.name)
    if n_dev is not None:
        assert int(n_dev.item()) == ref["n"]
    if g_dev is not None:
        g = g_dev.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
        harness.check_grad(g, ref, w, t_cpu, dloss=dl)
    return ref


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V", [1, 7, 8, 9, 33, 4095, 4096, 8200])
def test_small_and_unaligned_vocab(dtype, V):
    for N, a, red in ((1, 0.0, False), (3, 0.2, True), (5, 0.0, False)):
        w = wl.Workload(f"v{V}", 1, N, V, dtype, sigma=2.0, ignore_frac=0.2 if N > 3 else 0.0,
                        label_smoothing=a, reduce_loss=red, seed=11 + V + N)
        x = wl.logits(w)
        t = wl.targets(w)
        xd, td = x.to(DEV), t.to(DEV)
        n = torch.zeros(1, dtype=torch.int64, device=DEV)
        loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=a, reduce_loss=red, n_non_ignore_out=n)
        _compare(w, x, t, loss, xd, n)


@pytest.mark.parametrize("dtype,pad", [("bf16", 8), ("bf16", 3), ("f32", 4), ("f16", 16),
                                       ("bf16", 32000)])
def test_padded_rows(dtype, pad):
    w = wl.Workload("pad", 2, 5, 4000, dtype, sigma=2.0, label_smoothing=0.1, seed=31)
    x = wl.logits(w)
    buf = torch.zeros(2, 5, 4000 + pad, dtype=TDT[dtype])
    buf[:, :, :4000] = x
    t = wl.targets(w)
    bd = buf.to(DEV)
    view = bd[:, :, :4000]
    loss = pkg.ce_fwd_bwd(view, t.to(DEV), label_smoothing=0.1)
    _compare(w, buf, t, loss, None, strides=(5 * (4000 + pad), 4000 + pad))
    g = view.float().cpu().numpy().reshape(w.N, w.V)
    ref = harness.oracle_run(w, x, t)
    harness.check_grad(g, ref, w, t)
    # the padding is never touched
    assert torch.all(bd[:, :, 4000:].cpu() == 0)


@pytest.mark.parametrize("V", [4096, 32000])
def test_transposed_view(V):
    # storage (SQ, B, V), read as (B, SQ, V) through strides
    SQ, B = 6, 3
    w = wl.Workload("tr", SQ, B, V, "bf16", sigma=2.0, label_smoothing=0.1, seed=41)
    x = wl.logits(w)                # (SQ, B, V)
    t = wl.targets(w)               # (SQ, B)
    xd = x.to(DEV)
    td = t.to(DEV)
    v = xd.permute(1, 0, 2)         # (B, SQ, V), strides (V, B*V, 1)
    tv = td.t()                     # (B, SQ), strides (1, B)
    loss = pkg.ce_fwd_bwd(v, tv, label_smoothing=0.1)
    ref = oracle.ce(harness.storage_np(x), oracle.BF16, B, SQ, V, strides=(V, B * V),
                    targets=t.numpy().ravel(), target_strides=(1, B), label_smoothing=0.1)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], "bf16")
    g = v.float().cpu().numpy().reshape(B * SQ, V).astype(np.float64)
    # flattened rows of the (B, SQ) view: row b*SQ + s has target t[s, b]
    excess, _ = harness.grad_errors(g, ref["grad"], "bf16", np.ones(B * SQ), 0.1,
                                    t.t().contiguous().numpy().ravel())
    assert excess <= 0.0


@pytest.mark.parametrize("K", [2, 3, 5, 8, 16, 32])
def test_cluster_chunk_counts(K):
    w = wl.Workload("k", 1, 40, 24000, "bf16", sigma=2.0, label_smoothing=0.1, reduce_loss=True,
                    seed=50 + K)
    if K <= 16:
        harness.run_gpu_vs_oracle(w, force_path=2, num_vocab_chunks=K)
    harness.run_gpu_vs_oracle(w, force_path=3, num_vocab_chunks=K)
    harness.run_gpu_vs_oracle(w, force_path=4, num_vocab_chunks=K)


@pytest.mark.parametrize("name,K,tile_kb", [("c4_bsv65536_bf16_split8", 8, 0),
                                            ("c5_bsv128000_bf16_ls", 8, 0),
                                            ("c5_bsv128000_bf16_ls", 8, 16),
                                            ("c5_bsv128000_f32_ls", 5, 0),
                                            ("c2_sbv8192_bf16", 3, 0),
                                            ("c3h_bsv32000_f16_spiked", 32, 32)])
def test_stream_split_chunk_partials(name, K, tile_kb):
    """A split asked for on the stream kernel: each chunk of C = ceil(V/K)
    columns (rounded up to 16 bytes) streams as its own run of tiles and its
    partial {m, d, S, x_y} lands in the workspace; against the oracle's
    partials of the same columns (hyper-parallel #269 section 3.1: the
    per-slice max, sum-exp and target logit that the ranks exchange)."""
    w = wl.WORKLOADS[name].with_(dim0=1, dim1=48)
    x = wl.logits(w)
    t = wl.targets(w)
    opts = pkg.make_options(force_path=pkg.CE_PATH_STREAM, num_vocab_chunks=K, tune_tile_kb=tile_kb)
    xd = x.to(DEV)
    assert pkg.ce_plan_path(xd, opts)[0] == pkg.CE_PATH_STREAM
    vec = 16 // w.elem_bytes
    C = -(-(-(-w.V // K)) // vec) * vec
    nch = -(-w.V // C)
    assert pkg.ce_plan_path(xd, opts)[1] == nch
    ws = torch.zeros(pkg.ce_workspace_bytes(1, w.N, w.V, xd.dtype, opts), dtype=torch.uint8,
                     device=DEV)
    loss = pkg.ce_fwd_bwd(xd, t.to(DEV), label_smoothing=w.label_smoothing,
                          reduce_loss=w.reduce_loss, workspace=ws, opts=opts)
    assert pkg.ce_get_error(ws) == (0, 0)
    off = 256 + -(-w.N * 4 // 256) * 256
    part = ws[off:off + w.N * nch * 16].cpu().view(torch.float32).numpy().reshape(w.N, nch, 4)
    xv = x.float().numpy().reshape(w.N, w.V).astype(np.float64)
    tt = t.numpy().ravel()
    for r in range(w.N):
        if tt[r] == w.ignore_idx:
            continue
        for c in range(nch):
            k0, k1 = c * C, min(w.V, (c + 1) * C)
            ref = oracle.chunk_partials(xv[r], k0, k1, tt[r])
            m, d, S, xy = part[r, c].astype(np.float64)
            assert m == ref[0], (r, c)                            # max of stored values: exact
            assert abs(d - ref[1]) <= 1e-5 * ref[1], (r, c)
            assert abs(S - ref[2]) <= 1e-5 * np.abs(xv[r, k0:k1]).sum() + 1e-6, (r, c)
            assert xy == ref[3], (r, c)                           # the target logit, exact
    ref = harness.oracle_run(w, x, t, dloss=np.array([1.0]) if w.reduce_loss else None)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, name)
    harness.check_grad(xd.float().cpu().numpy(), ref, w, t,
                       dloss=np.array([1.0]) if w.reduce_loss else None)


@pytest.mark.parametrize("V,dtype", [(20011, "bf16"), (16389, "f16"), (10007, "f32"),
                                     (7, "bf16"), (33, "f16"), (4095, "bf16"), (3, "f32")])
def test_stream_edges_targets_at_the_edges(V, dtype):
    """Rows off the 16-byte grid on the stream kernel: the ring takes each
    row's aligned body, threads take the head and tail elements one each.
    Row starts cycle through the offsets from a 16-byte boundary (odd
    widths), and targets sit on the first and last elements of each row, so
    the target is a head, body or tail element; tiny widths have no body."""
    N = 48
    w = wl.Workload(f"edges{V}", 1, N, V, dtype, sigma=2.0, ignore_frac=0.1, label_smoothing=0.1,
                    seed=V + 5)
    x = wl.logits(w)
    t = wl.targets(w)
    tf = t.view(-1)
    for r in range(0, 16):
        if tf[r] != -100:
            tf[r] = r % min(8, V) if r < 8 else V - 1 - (r % min(8, V))
    opts = pkg.make_options(force_path=pkg.CE_PATH_STREAM)
    xd = x.to(DEV)
    assert pkg.ce_plan_path(xd, opts)[0] == pkg.CE_PATH_STREAM
    rng = np.random.default_rng(V)
    dl = rng.uniform(0.5, 2.0, N).astype(np.float32).astype(np.float64)
    loss = pkg.ce_fwd_bwd(xd, t.to(DEV), label_smoothing=0.1,
                          dloss=torch.tensor(dl, dtype=torch.float32, device=DEV), opts=opts)
    ref = harness.oracle_run(w, x, t, dloss=dl)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], dtype, w.name)
    g = xd.float().cpu().numpy().reshape(N, V)
    assert np.all(g[wl.ignored_rows(w)] == 0.0)
    harness.check_grad(g, ref, w, t, dloss=dl)


def test_empty_chunks():
    # V = 16 bf16 over 8 CTAs: 16-byte chunks of 8 columns leave six CTAs empty
    w = wl.Workload("e", 1, 7, 16, "bf16", sigma=3.0, seed=61)
    harness.run_gpu_vs_oracle(w, force_path=2, num_vocab_chunks=8)
    w = wl.Workload("e", 1, 7, 40, "f32", sigma=3.0, seed=62)
    harness.run_gpu_vs_oracle(w, force_path=2, num_vocab_chunks=16)


@pytest.mark.parametrize("path", [0, 1, 3, 4, 5, 6])
def test_all_ignored_mean_is_nan(path):
    x = torch.randn(3, 4, 1024, device=DEV).to(torch.bfloat16)
    t = torch.full((3, 4), -100, dtype=torch.int64, device=DEV)
    n = torch.ones(1, dtype=torch.int64, device=DEV)
    loss = pkg.ce_fwd_bwd(x, t, reduce_loss=True, n_non_ignore_out=n, force_path=path)
    assert math.isnan(loss.item()) and int(n.item()) == 0
    assert torch.all(x == 0)


@pytest.mark.parametrize("path", [0, 1, 2, 3, 4, 5, 6])
def test_out_of_range_target_sets_error(path):
    w = wl.Workload("oor", 1, 6, 8192, "bf16", sigma=2.0, ignore_frac=0.0, seed=71)
    x = wl.logits(w)
    t = wl.targets(w)
    t[0, 2] = 8192
    t[0, 4] = -7
    xd, td = x.to(DEV), t.to(DEV)
    ws = torch.empty(pkg.ce_workspace_bytes(1, 6, 8192, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    loss = pkg.ce_fwd_bwd(xd, td, workspace=ws, force_path=path)
    st, err = pkg.ce_get_error(ws)
    assert err & 1 and st == 6
    lc = loss.cpu().numpy()
    assert math.isnan(lc[2]) and math.isnan(lc[4])
    assert torch.all(xd[0, 2] == 0) and torch.all(xd[0, 4] == 0)
    ref = harness.oracle_run(w, x, t)
    keep = [0, 1, 3, 5]
    harness.check_loss(lc[keep], ref["loss"][keep], "bf16")
    # a later clean pass on the same workspace clears the error word
    loss = pkg.ce_fwd_bwd(x.to(DEV), wl.targets(w).to(DEV), workspace=ws, force_path=path)
    assert pkg.ce_get_error(ws) == (0, 0)


def test_non_negative_ignore_index():
    w = wl.Workload("ig", 1, 9, 512, "f32", sigma=1.0, ignore_frac=0.0, seed=81)
    x = wl.logits(w)
    t = wl.targets(w)
    t[0, 3] = 5
    w2 = w.with_(ignore_idx=5)
    xd = x.to(DEV)
    loss = pkg.ce_fwd_bwd(xd, t.to(DEV), ignore_idx=5)
    ref = harness.oracle_run(w2, x, t)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], "f32")
    assert loss[3].item() == 0.0 and torch.all(xd[0, 3] == 0)


def test_zero_rows():
    x = torch.empty(0, 4, 4096, dtype=torch.bfloat16, device=DEV)
    t = torch.empty(0, 4, dtype=torch.int64, device=DEV)
    loss = pkg.ce_fwd_bwd(x, t, reduce_loss=True)
    assert math.isnan(loss.item())
    loss = pkg.ce_fwd_bwd(x, t, reduce_loss=False)
    assert loss.numel() == 0


@pytest.mark.parametrize("name,path", [("c5_bsv128000_bf16_ls", 0), ("c3_bsv32000_bf16_spiked", 0),
                                       ("c2_sbv8192_bf16", 0), ("c4_bsv65536_bf16_split8", 3),
                                       ("c5_bsv128000_bf16_ls", 2), ("c1_bsv4096_f32", 1),
                                       ("c1_bsv4096_f32", 5), ("c1_bsv4096_f32", 6),
                                       ("c5_bsv128000_bf16_ls", 6)])
def test_fwd_only_matches(name, path):
    w = wl.WORKLOADS[name]
    x = wl.logits(w)
    t = wl.targets(w)
    xd, td = x.to(DEV), t.to(DEV)
    lse = torch.empty(w.N, dtype=torch.float32, device=DEV)
    loss = pkg.ce_fwd_only(xd, td, label_smoothing=w.label_smoothing, reduce_loss=False,
                           lse_out=lse, force_path=path)
    assert torch.equal(xd.cpu(), x)  # logits untouched
    ref = harness.oracle_run(w.with_(reduce_loss=False), x, t, want_grad=False)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype)
    lse_ref = ref["lse"]
    lg = lse.cpu().numpy().astype(np.float64)
    ok = ~np.isnan(lse_ref)
    assert np.all(np.isnan(lg[~ok]))
    assert np.max(np.abs(lg[ok] - lse_ref[ok]) / np.maximum(np.abs(lse_ref[ok]), 1)) <= 1e-5
    # forward-only losses equal the fused pass's losses bit for bit on the fused paths
    loss2 = pkg.ce_fwd_bwd(xd.clone(), td, label_smoothing=w.label_smoothing, force_path=path)
    if path != 3:
        assert torch.equal(loss, loss2)


@pytest.mark.parametrize("name,path", [("c5_bsv128000_bf16_ls", 0), ("c2_sbv8192_bf16", 0),
                                       ("c2_sbv8192_bf16", 1), ("c4_bsv65536_bf16_split8", 3),
                                       ("c5_bsv128000_bf16_ls", 6)])
def test_mean_is_deterministic(name, path):
    w = wl.WORKLOADS[name]
    x = wl.logits(w).to(DEV)
    t = wl.targets(w).to(DEV)
    vals = []
    for _ in range(10):
        loss = pkg.ce_fwd_bwd(x.clone(), t, label_smoothing=w.label_smoothing, reduce_loss=True,
                              force_path=path)
        vals.append(loss.cpu().numpy().tobytes())
    assert len(set(vals)) == 1


def test_full_size_sampled_rows():
    """The throughput workload (4, 4096, 128000) bf16 in the launch
    configuration the bench times: the mean against the oracle over all rows,
    and the gradient of sampled rows element by element."""
    w = wl.WORKLOADS["c5t_bsv128000_bf16"]
    x = wl.logits(w)
    t = wl.targets(w)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(w.N, 48, replace=False))
    rows = np.unique(np.concatenate([rows, wl.ignored_rows(w)[:4], [0, w.N - 1]]))
    xd = x.to(DEV)
    td = t.to(DEV)
    n = torch.zeros(1, dtype=torch.int64, device=DEV)
    loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=w.label_smoothing, reduce_loss=True,
                          n_non_ignore_out=n)
    g_rows = xd.view(w.N, w.V)[torch.as_tensor(rows, device=DEV)].float().cpu().numpy()
    del xd
    ref_all = harness.oracle_run(w, x, t, want_grad=False)
    assert int(n.item()) == ref_all["n"]
    harness.check_loss(loss.cpu().numpy(), ref_all["loss"], "bf16", "full-size mean")
    # per-row oracle on the sampled rows, scale dloss/n of the full pass
    sub = x.view(w.N, w.V)[torch.as_tensor(rows)].contiguous()
    tsub = t.view(-1)[torch.as_tensor(rows)].contiguous()
    scale = np.full(len(rows), 1.0 / ref_all["n"])
    ref = oracle.ce(harness.storage_np(sub), oracle.BF16, 1, len(rows), w.V,
                    targets=tsub.numpy(), label_smoothing=w.label_smoothing, dloss=scale)
    excess, _ = harness.grad_errors(g_rows.astype(np.float64), ref["grad"], "bf16", scale,
                                    w.label_smoothing, tsub.numpy())
    assert excess <= 0.0


@pytest.mark.parametrize("V,dtype,tile_kb,stages", [(12000, "bf16", 0, 0), (16384, "bf16", 0, 0),
                                                    (8192, "f32", 0, 0), (5000, "f32", 0, 0),
                                                    (8192, "bf16", 16, 6), (4096, "f16", 32, 6),
                                                    (2048, "bf16", 16, 12)])
def test_warp_path_tiles(V, dtype, tile_kb, stages):
    """Rows of up to one 16 or 32 KB tile on the warp-per-row path: every
    consumer warp owns its tiles; rows, ignored rows and tiles do not line up."""
    for N, a, red in ((1, 0.1, True), (37, 0.0, False), (301, 0.1, True)):
        w = wl.Workload(f"warp{V}", 1, N, V, dtype, sigma=2.0, ignore_frac=0.15,
                        label_smoothing=a, reduce_loss=red, seed=V + N)
        opts = pkg.make_options(force_path=5, tune_tile_kb=tile_kb, tune_stages=stages)
        x = wl.logits(w)
        t = wl.targets(w)
        xd, td = x.to(DEV), t.to(DEV)
        ws = torch.empty(pkg.ce_workspace_bytes(1, N, V, xd.dtype, opts), dtype=torch.uint8,
                         device=DEV)
        n = torch.zeros(1, dtype=torch.int64, device=DEV)
        loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=a, reduce_loss=red, n_non_ignore_out=n,
                              workspace=ws, opts=opts)
        assert pkg.ce_get_error(ws) == (0, 0)
        _compare(w, x, t, loss, xd, n)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("V", [4096, 8192, 12000])
def test_warp_rows_wide_range(dtype, V):
    """16-bit rows on the warp path with extreme ranges: spikes of +60 to
    +120 away from and inside the first vectors, hugely negative first
    vectors and single elements, a uniform shift of -1000; against the
    oracle."""
    N = 24
    w = wl.Workload("warp_range", 1, N, V, dtype, sigma=2.0, label_smoothing=0.1,
                    reduce_loss=False, seed=7700 + V)
    x = wl.logits(w).float()
    low = -1e30 if dtype == "bf16" else -60000.0
    c = 3001
    for r, spike in enumerate([100.0, 100.0, 60.0, 80.0, 88.5, 89.0, 120.0]):
        x[0, r, c] += spike
    x[0, 7, 5] += 100.0                  # in lane 0's first vector
    x[0, 8, 0:8] = low                   # lane 0's first vector
    x[0, 9, 0:256] = low                 # every lane's first vector
    x[0, 10, :] -= 1000.0                # a uniform shift
    x[0, 11, c] = low                    # one very low element
    x = x.to(TDT[dtype])
    t = wl.targets(w)
    t[0, :12] = torch.arange(12) * 97 + 300  # away from the edited columns
    xd, td = x.to(DEV), t.to(DEV)
    assert pkg.ce_plan_path(xd)[0] == pkg.CE_PATH_WARP
    ws = torch.empty(pkg.ce_workspace_bytes(1, N, V, xd.dtype), dtype=torch.uint8, device=DEV)
    loss = pkg.ce_fwd_bwd(xd, td, label_smoothing=0.1, reduce_loss=False, workspace=ws)
    assert pkg.ce_get_error(ws) == (0, 0)
    _compare(w, x, t, loss, xd)


@pytest.mark.parametrize("grad", [True, False])
def test_row_counter_left_zeroed(grad):
    """The stream kernel hands out rows past each CTA's first two from a
    counter in the workspace; every pass must leave it (and the count of CTAs
    done with it) at zero, so a pass that follows without a count kernel in
    between -- the chunks of the lm_head pass -- starts from row 0 again."""
    w = wl.WORKLOADS["c3_bsv32000_bf16_spiked"]  # 1024 rows: more than the CTAs
    dev = torch.device("cuda")
    x = wl.logits(w).to(dev)
    t = wl.targets(w).to(dev)
    assert pkg.ce_plan_path(x)[0] == pkg.CE_PATH_STREAM
    ws = torch.full((pkg.ce_workspace_bytes(w.dim0, w.dim1, w.V, x.dtype),), 0x5A,
                    dtype=torch.uint8, device=dev)  # garbage before the first pass
    first = None
    for _ in range(2):
        xi = x.clone()
        if grad:
            loss = pkg.ce_fwd_bwd(xi, t, reduce_loss=False, workspace=ws)
        else:
            loss = pkg.ce_fwd_only(xi, t, reduce_loss=False, workspace=ws)
        words = ws[40:48].cpu().numpy().view(np.uint32)
        assert words.tolist() == [0, 0], words
        st, err = pkg.ce_get_error(ws)
        assert st == 0 and err == 0
        if first is None:
            first = (loss.clone(), xi)
        else:  # the second pass over the same workspace gives the same results
            assert torch.equal(loss, first[0])
            assert torch.equal(xi, first[1])


@pytest.mark.parametrize("N", [1, 151, 152, 153, 303, 304, 305, 700])
@pytest.mark.parametrize("reduce", [True, False])
def test_stream_row_counts(N, reduce):
    """Row counts around one and two grids of the stream kernel (152 CTAs on
    a GB300): CTAs with one row, with their two first rows only, and the first
    rows claimed from the shared counter -- every row is computed once, and
    matches the oracle."""
    w = wl.WORKLOADS["c5_bsv128000_bf16_ls"].with_(
        name=f"stream_rows_{N}", dim0=1, dim1=N, V=20000, reduce_loss=reduce, seed=3000 + N)
    x = wl.logits(w)
    assert pkg.ce_plan_path(x.to(DEV))[0] == pkg.CE_PATH_STREAM
    harness.run_gpu_vs_oracle(w, per_row_dloss=not reduce)


def test_bounded_wait_reports_timeout():
    """Failure detection without a fault: the bounded wait the kernels use,
    left to run out on a barrier nothing completes, reports CE_DEVERR_TIMEOUT
    through the workspace, and the GPU takes the next pass normally."""
    import time
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    t0 = time.time()
    pkg.ce_wait_timeout_probe(ws)
    st, err = pkg.ce_get_error(ws)
    waited = time.time() - t0
    assert err == 0x2 and st == 7, (st, err)  # CE_DEVERR_TIMEOUT, CE_ERR_DEVICE_TIMEOUT
    assert 1.0 < waited < 30.0
    assert "gave up" in pkg.ce_status_string(st)
    w = wl.WORKLOADS["c2_sbv8192_bf16"]
    harness.run_gpu_vs_oracle(w)  # the context is still usable


@pytest.mark.parametrize("V,path", [(1 << 20, pkg.CE_PATH_STREAM), ((1 << 20) + 3, pkg.CE_PATH_STREAM),
                                    (256000, pkg.CE_PATH_STREAM), (200000, pkg.CE_PATH_STREAM),
                                    (200003, pkg.CE_PATH_STREAM)])
@pytest.mark.parametrize("reduce", [True, False])
def test_very_wide_rows(V, path, reduce):
    """Rows of a million columns (2 MB of bf16 each: 64 ring tiles per pass on
    the stream path; an odd width goes to the plain-load kernel), and rows of
    16 and 13 tiles (the last one partial) -- all wide enough for pass 2 to
    take the ring's last tiles from shared memory -- against the oracle."""
    w = wl.WORKLOADS["c5_bsv128000_bf16_ls"].with_(
        name=f"wide_{V}", dim0=2, dim1=12, V=V, reduce_loss=reduce, seed=4000 + V % 97)
    x = wl.logits(w)
    assert pkg.ce_plan_path(x.to(DEV))[0] == path
    harness.run_gpu_vs_oracle(w, per_row_dloss=not reduce)
    if V % 8:  # the plain-load kernel on the same odd-width rows
        harness.run_gpu_vs_oracle(w, force_path=pkg.CE_PATH_VECROW, per_row_dloss=not reduce)


def test_warp_path_two_tiles_by_default():
    """From 8192 rows on, the planner gives each consumer warp of the
    warp-per-row kernel two 16 KB tiles (a 12-deep ring): many rows per warp,
    tiles reused in turn, against the oracle."""
    w = wl.Workload("warp_many_rows", 1, 9000, 8192, "bf16", sigma=2.0, ignore_frac=0.05,
                    label_smoothing=0.1, reduce_loss=True, seed=9000)
    assert pkg.ce_plan_path(wl.logits(w).to(DEV))[0] == pkg.CE_PATH_WARP
    harness.run_gpu_vs_oracle(w)


@pytest.mark.parametrize("V,dtype,a,reduce,ignore", [(100277, "bf16", 0.1, True, 0.1),
                                                     (50257, "f16", 0.0, False, 0.2),
                                                     (100003, "f32", 0.2, True, 0.0),
                                                     (16387, "bf16", 0.0, False, 0.05)])
@pytest.mark.parametrize("path", [pkg.CE_PATH_AUTO, pkg.CE_PATH_TWO_STAGE, pkg.CE_PATH_VECROW])
def test_unaligned_rows(V, dtype, a, reduce, ignore, path):
    """Odd widths put every row at its own offset from a 16-byte boundary.
    The planner sends rows over 32 KB to the stream kernel (the aligned body
    through the TMA ring, the head and tail elements one per thread), and
    narrower ones to the plain-load kernel (a scalar head, 16-byte vectors,
    a scalar tail), which also takes the wide ones when forced; the two-stage
    kernels read each chunk the same way (several chunks per row, the last
    one ragged)."""
    w = wl.Workload(f"unaligned_{V}", 2, 17, V, dtype, sigma=2.0, ignore_frac=ignore,
                    label_smoothing=a, reduce_loss=reduce, seed=V % 1000)
    if path == pkg.CE_PATH_AUTO:
        want = pkg.CE_PATH_STREAM if V * w.elem_bytes > 32 * 1024 else pkg.CE_PATH_VECROW
        assert pkg.ce_plan_path(wl.logits(w).to(DEV))[0] == want
    harness.run_gpu_vs_oracle(w, force_path=path, per_row_dloss=not reduce)


@pytest.mark.parametrize("threads,cap", [(256, 0), (512, 1), (256, 1), (1024, 0), (32, 0), (32, 1)])
def test_vecrow_shapes(threads, cap):
    """The plain-load kernel's other shapes on 40 KB rows: a CTA of 256
    threads (three per SM) or 1024 (one per SM), a warp per row (32), and
    grids capped to one CTA per SM, so each CTA or warp takes many rows."""
    w = wl.Workload("vecrow_shapes", 1, 700, 20011, "bf16", sigma=2.0, ignore_frac=0.1,
                    label_smoothing=0.1, reduce_loss=True, seed=threads + cap)
    x = wl.logits(w)
    t = wl.targets(w)
    ref = harness.oracle_run(w, x, t)
    xd = x.to(DEV)
    opts = pkg.make_options(force_path=pkg.CE_PATH_VECROW, tune_threads=threads,
                            tune_ctas_per_sm=cap)
    loss = pkg.ce_fwd_bwd(xd, t.to(DEV), label_smoothing=0.1, reduce_loss=True, opts=opts)
    harness.check_loss(loss.cpu().numpy().reshape(-1), ref["loss"], "bf16")
    g = xd.float().cpu().numpy().reshape(w.N, w.V).astype(np.float64)
    harness.check_grad(g, ref, w, t)


@pytest.mark.parametrize("K", [3, 7, 16])
def test_unaligned_rows_short_chunks(K):
    """Chunks shorter than a 16-byte vector (37 bf16 columns in up to 16
    chunks of 3): some chunks are all head, some hold no whole vector."""
    w = wl.Workload("short_chunks", 1, 11, 37, "bf16", sigma=2.0, ignore_frac=0.2,
                    label_smoothing=0.1, reduce_loss=True, seed=37 + K)
    harness.run_gpu_vs_oracle(w, force_path=pkg.CE_PATH_TWO_STAGE, num_vocab_chunks=K)


@pytest.mark.parametrize("dtype,shift", [("bf16", 1), ("bf16", 5), ("f16", 3), ("f32", 1)])
@pytest.mark.parametrize("path", [pkg.CE_PATH_AUTO, pkg.CE_PATH_TWO_STAGE, pkg.CE_PATH_VECROW])
def test_shifted_view_rows(dtype, shift, path):
    """An aligned width read through a view that starts `shift` elements
    into each padded row: the rows leave the 16-byte grid, the stream kernel
    (aligned body by TMA, head and tail by threads) takes them, or forced the
    plain-load or two-stage kernels, and the padding on both sides stays
    untouched."""
    V, pad = 32000, 9
    w = wl.Workload("shifted", 2, 5, V, dtype, sigma=2.0, label_smoothing=0.1, seed=50 + shift)
    x = wl.logits(w)
    buf = torch.zeros(2, 5, V + pad, dtype=TDT[dtype])
    buf[:, :, shift:shift + V] = x
    t = wl.targets(w)
    bd = buf.to(DEV)
    view = bd[:, :, shift:shift + V]
    if path == pkg.CE_PATH_AUTO:
        assert pkg.ce_plan_path(view)[0] == pkg.CE_PATH_STREAM
    loss = pkg.ce_fwd_bwd(view, t.to(DEV), label_smoothing=0.1, force_path=path)
    ref = harness.oracle_run(w, x, t)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], dtype, "shifted")
    g = view.float().cpu().numpy().reshape(w.N, V).astype(np.float64)
    harness.check_grad(g, ref, w, t)
    host = bd.cpu()
    assert torch.all(host[:, :, :shift] == 0)
    assert torch.all(host[:, :, shift + V:] == 0)
