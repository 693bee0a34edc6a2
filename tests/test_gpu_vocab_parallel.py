"""Vocabulary-parallel steps (partials per shard, combine, per-shard
backward) over shards held as separate tensors on one GPU, against the CPU
oracle on the unsharded rows (hyper-parallel #269 section 3.1: the combine of
ceil(V/tp) slices must reproduce the unsplit cross-entropy)."""
import numpy as np
import pytest
import torch

import oracle
import vocabulary_cross_entropy_pass_gb300 as pkg
from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _shards(x, R):
    V = x.shape[-1]
    c = -(-V // R)  # ceil(V/R); the last shard is shorter
    return [x[..., k * c:min(V, (k + 1) * c)].contiguous() for k in range(R) if k * c < V]


@pytest.mark.parametrize("name,R", [("c4_bsv65536_bf16_split8", 8), ("c5_bsv128000_bf16_ls", 8),
                                    ("c5_bsv128000_f32_ls", 3), ("c1_bsv4096_f32", 2),
                                    ("c3h_bsv32000_f16_spiked", 5)])
def test_vocab_parallel_matches_unsharded(name, R):
    w = wl.WORKLOADS[name]
    x = wl.logits(w)
    t = wl.targets(w)
    dl = np.array([1.0]) if w.reduce_loss else None
    ref = harness.oracle_run(w, x, t, dloss=dl)
    td = t.to(DEV)
    shards = [s.to(DEV) for s in _shards(x, R)]
    loss, grads = pkg.vocab_parallel_cross_entropy(shards, td, label_smoothing=w.label_smoothing,
                                                   reduce_loss=w.reduce_loss)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], w.dtype, name)
    g = torch.cat([gr.float().cpu() for gr in grads], dim=-1).numpy().reshape(w.N, w.V)
    harness.check_grad(g, ref, w, t, dloss=dl)


def test_vocab_parallel_uneven_unaligned_shards():
    # V = 1001 bf16 over 4 shards of 251 columns: no shard row is 16-byte aligned
    w = wl.Workload("vp", 2, 33, 1001, "bf16", sigma=2.0, ignore_frac=0.2, label_smoothing=0.2,
                    reduce_loss=True, seed=77)
    x = wl.logits(w)
    t = wl.targets(w)
    ref = harness.oracle_run(w, x, t, dloss=np.array([1.0]))
    shards = [s.to(DEV) for s in _shards(x, 4)]
    loss, grads = pkg.vocab_parallel_cross_entropy(shards, t.to(DEV), label_smoothing=0.2,
                                                   reduce_loss=True, inplace_grad=False)
    harness.check_loss(loss.cpu().numpy(), ref["loss"], "bf16")
    g = torch.cat([gr.float().cpu() for gr in grads], dim=-1).numpy().reshape(w.N, w.V)
    harness.check_grad(g, ref, w, t, dloss=np.array([1.0]))


def test_vocab_parallel_partials_combine_lse():
    w = wl.WORKLOADS["c2_sbv8192_bf16"]
    x = wl.logits(w)
    t = wl.targets(w)
    ref = harness.oracle_run(w.with_(reduce_loss=False), x, t, want_grad=False)
    shards = [s.to(DEV) for s in _shards(x, 4)]
    offs = [0, 2048, 4096, 6144, 8192]
    part = torch.stack([pkg.ce_vp_partials(s, t.to(DEV), offs[k]) for k, s in enumerate(shards)])
    n = torch.empty(1, dtype=torch.int64, device=DEV)
    loss, lse = pkg.ce_vp_combine(part, offs, t.to(DEV), label_smoothing=0.1, n_non_ignore_out=n)
    assert int(n.item()) == ref["n"]
    ok = ~np.isnan(ref["lse"])
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isnan(lg[~ok]))
    assert np.max(np.abs(lg[ok] - ref["lse"][ok]) / np.abs(ref["lse"][ok])) <= 1e-5
    harness.check_loss(loss.cpu().numpy(), ref["loss"], "bf16")


@pytest.mark.parametrize("dtype,V,cuts", [("bf16", 64000, [0, 20000, 40000, 64000]),
                                          ("f16", 50000, [0, 8192, 50000]),
                                          ("f32", 24003, [0, 4096, 12196, 24003]),
                                          ("bf16", 30000, [0, 8191, 30000])])
def test_vp_partials_against_oracle(dtype, V, cuts):
    """Step 1 on shards on and off the 16-byte grid, of 16 KB and more and
    less: each row's {m, d, S, x_y} against the oracle's partial of the same
    columns (hyper-parallel #269 section 3.1), ignored rows {-inf, 0, 0, 0},
    targets inside and outside each shard."""
    w = wl.Workload("vp_part", 3, 101, V, dtype, sigma=2.0, ignore_frac=0.2, seed=V + len(cuts))
    x = wl.logits(w)
    t = wl.targets(w)
    td = t.to(DEV)
    xv = x.float().numpy().reshape(w.N, V).astype(np.float64)
    tt = t.numpy().ravel()
    for k0, k1 in zip(cuts[:-1], cuts[1:]):
        part = pkg.ce_vp_partials(x[..., k0:k1].contiguous().to(DEV), td, k0).cpu().numpy()
        part = part.reshape(w.N, 4).astype(np.float64)
        for r in range(w.N):
            m, d, S, xy = part[r]
            if tt[r] == w.ignore_idx:
                assert m == -np.inf and d == 0.0 and S == 0.0 and xy == 0.0, (k0, r)
                continue
            ref = oracle.chunk_partials(xv[r], k0, k1, tt[r])
            assert m == ref[0], (k0, r)                            # max of stored values: exact
            assert abs(d - ref[1]) <= 1e-5 * ref[1], (k0, r)
            assert abs(S - ref[2]) <= 1e-5 * np.abs(xv[r, k0:k1]).sum() + 1e-6, (k0, r)
            assert xy == ref[3], (k0, r)                           # the target logit, exact

