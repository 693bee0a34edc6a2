"""Vocabulary-parallel steps (partials per shard, combine, per-shard
backward) over shards held as separate tensors on one GPU, against the CPU
oracle on the unsharded rows (hyper-parallel #269 section 3.1: the combine of
ceil(V/tp) slices must reproduce the unsplit cross-entropy)."""
import numpy as np
import pytest
import torch

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
