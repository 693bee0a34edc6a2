"""lm_head + cross-entropy chunked over rows against the CPU oracle of the
same dataflow: bf16/fp16 take this library's tcgen05 GEMM with the
cross-entropy statistics in its epilogue, then the backward from lse; fp32
(and hidden sizes off a multiple of 8) a cuBLAS GEMM and the fused pass; the
gradient GEMMs are cuBLAS's.

Tolerances: the loss as for the pass, plus one unit in the last place of the
row's target logit (the GEMM's float32 sum and the oracle's double sum may
round a logit to neighbouring values of the storage dtype); the gradients as a
GEMM of the compared logits gradient: 2^-7 (bf16/fp16) or 1e-5 (fp32) of
sum |dlogits| |other operand|, plus the final rounding of grad_hidden."""
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


@pytest.mark.parametrize("N,H,V,dtype,chunk,a,red", [
    (333, 192, 4000, "bf16", 128, 0.1, True),     # warp path per chunk, ragged last chunk
    (200, 96, 20000, "bf16", 64, 0.0, False),     # stream path per chunk
    # stream path, chunks of more rows than CTAs: rows are claimed from the
    # shared counter, which each chunk's pass leaves zeroed for the next
    (1200, 64, 20000, "bf16", 400, 0.1, True),
    (100, 64, 3000, "f32", 37, 0.1, False),
    (150, 128, 6000, "f16", 1000, 0.0, True),     # one chunk
    # the tensor-core GEMM: 2 x 63 tiles of 128 x 256 per chunk (several per
    # CTA, both accumulators in turn) and 8 K steps (twice round the ring)
    (777, 512, 16000, "bf16", 256, 0.1, True),
    (300, 256, 4001, "bf16", 300, 0.0, False),    # odd vocabulary: padded logits rows
    (260, 320, 5000, "f16", 130, 0.1, False),     # 5 K steps, the last half out of range
    (200, 100, 3000, "bf16", 100, 0.1, True),     # hidden size off 8: the cuBLAS path
    # one-CTA kernel (64-row chunks), 2 K steps of which the second is mostly
    # out of range, a last vocabulary tile of one column
    (64, 72, 4097, "bf16", 64, 0.1, True),
    (300, 128, 200, "f16", 300, 0.0, False),      # paired kernel, the vocabulary inside one tile
])
def test_linear_ce_matches_oracle(N, H, V, dtype, chunk, a, red):
    rng = np.random.default_rng(N + V)
    h32 = rng.standard_normal((N, H)).astype(np.float32)
    w32 = (rng.standard_normal((V, H)) / np.sqrt(H) * 2).astype(np.float32)
    h = torch.from_numpy(h32).to(TDT[dtype])
    w = torch.from_numpy(w32).to(TDT[dtype])
    t = torch.from_numpy(rng.integers(0, V, N).astype(np.int64))
    t[rng.permutation(N)[: N // 10]] = -100
    dl = np.array([1.0]) if red else rng.uniform(0.5, 2.0, N).astype(np.float32)
    ref = oracle.linear_ce(harness.storage_np(h), harness.storage_np(w), harness.CODE[dtype], N, H,
                           V, t.numpy(), label_smoothing=a, reduce_loss=red,
                           dloss=dl.astype(np.float64))
    n = torch.zeros(1, dtype=torch.int64, device=DEV)
    loss, gh, gw = pkg.ce_linear_fwd_bwd(h.to(DEV), w.to(DEV), t.to(DEV), label_smoothing=a,
                                         reduce_loss=red,
                                         dloss=torch.tensor(dl, dtype=torch.float32, device=DEV),
                                         chunk_rows=chunk, n_non_ignore_out=n)
    assert int(n.item()) == ref["n"]
    hd = h.to(torch.float64).numpy()
    wd = w.to(torch.float64).numpy()
    logits = hd @ wd.T
    tt = t.numpy()
    kept = tt != -100
    # loss: the pass's tolerance plus one ulp of the target logit
    got = loss.cpu().numpy().astype(np.float64)
    if red:
        slack = np.max(harness.ulp(np.abs(logits[kept, tt[kept]]), dtype)) if dtype != "f32" else 0.0
        assert abs(got[0] - ref["loss"][0]) <= harness.LOSS_TOL[dtype] * max(1, abs(ref["loss"][0])) + slack
    else:
        slack = np.zeros(N)
        if dtype != "f32":
            slack[kept] = harness.ulp(np.abs(logits[kept, tt[kept]]), dtype) * 2
        err = np.abs(got - ref["loss"]) - harness.LOSS_TOL[dtype] * np.maximum(np.abs(ref["loss"]), 1)
        assert np.all(err <= slack)
    rel = 2.0 ** -7 if dtype != "f32" else 1e-5
    bound_h = rel * (np.abs(ref["dlogits"]) @ np.abs(wd)) + 1e-6 * np.abs(wd).sum(axis=0)
    ghd = gh.to(torch.float64).cpu().numpy()
    if dtype != "f32":
        bound_h = bound_h + harness.ulp(ref["grad_hidden"], dtype)
    assert np.all(np.abs(ghd - ref["grad_hidden"]) <= bound_h)
    bound_w = rel * (np.abs(ref["dlogits"]).T @ np.abs(hd)) + 1e-6 * np.abs(hd).sum(axis=0)
    gwd = gw.to(torch.float64).cpu().numpy()
    assert np.all(np.abs(gwd - ref["grad_weight"]) <= bound_w)


def test_linear_ce_grad_weight_accumulates():
    rng = np.random.default_rng(5)
    N, H, V = 64, 32, 512
    h = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)).to(DEV).to(torch.bfloat16)
    w = torch.from_numpy((rng.standard_normal((V, H)) * 0.3).astype(np.float32)).to(DEV).to(torch.bfloat16)
    t = torch.from_numpy(rng.integers(0, V, N).astype(np.int64)).to(DEV)
    _, _, g1 = pkg.ce_linear_fwd_bwd(h, w, t, grad_hidden=None, chunk_rows=20)
    acc = g1.clone()
    pkg.ce_linear_fwd_bwd(h, w, t, grad_hidden=None, grad_weight=acc, chunk_rows=20)
    assert torch.allclose(acc, 2 * g1, rtol=1e-6, atol=1e-7)
