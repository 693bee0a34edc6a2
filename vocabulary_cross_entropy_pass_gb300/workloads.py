"""Seeded synthetic inputs for the cross-entropy pass.

This module draws random numbers and nothing else: it holds none of the
cross-entropy arithmetic, so both the GPU tests and the CPU oracle can take
their inputs from it.  The pages measure on no public dataset; the shapes
below are the typical shapes listed in the TENPU "Parallel Cross Entropy"
issue (section 5, performance data), with value spreads, ignore fractions and
smoothing factors chosen per workload.

Recipe (the same on every machine):
  * logits are drawn row block by row block (64 flattened rows per block,
    row r = i*dim1 + j); block b uses ``numpy.random.default_rng([seed, b])``
    and ``standard_normal(float32) * sigma``; a chosen 1% of rows (spiked
    workloads) get +spike at one uniform column, in float32;
  * the float32 values are cast to the storage dtype with torch's
    round-to-nearest-even conversion;
  * targets are uniform in [0, V) from ``default_rng([seed, 1 << 20])``;
    exactly floor(p * N) rows, picked by a seeded permutation, are set to
    ``ignore_idx``.

Any row block can be regenerated alone, so a test at full size can rebuild
the rows it samples without holding the whole tensor on the host.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROW_BLOCK = 64
_TARGET_STREAM = 1 << 20
_SPIKE_STREAM = 1 << 21
_IGNORE_STREAM = 1 << 22

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dim0: int
    dim1: int
    V: int
    dtype: str                 # "f32" | "bf16" | "f16"
    layout: str = "bsv"        # "bsv": (B, SQ, V); "sbv": (SQ, B, V)
    sigma: float = 1.0
    ignore_frac: float = 0.1
    spike_frac: float = 0.0
    spike: float = 20.0
    label_smoothing: float = 0.0
    reduce_loss: bool = False
    seed: int = 1000
    vocab_chunks: int = 0      # 0: the library picks; K > 0 forces K vocabulary chunks
    ignore_idx: int = -100

    @property
    def N(self) -> int:
        return self.dim0 * self.dim1

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def logits_bytes(self) -> int:
        return self.N * self.V * self.elem_bytes

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workload families: (2,128,4096) fp32; (SQ=256,B=4,8192) bf16 in
# (SQ,B,V) layout; (2,512,32000) bf16 with spiked rows and its fp16 twin;
# (2,256,65536) bf16 split into 8 vocabulary chunks; (1,512,128000) bf16/fp32
# for correctness and (4,4096,128000) bf16 for throughput.
WORKLOADS = {
    "c1_bsv4096_f32": Workload("c1_bsv4096_f32", 2, 128, 4096, "f32", "bsv", 1.0, 0.10,
                               seed=1001),
    "c2_sbv8192_bf16": Workload("c2_sbv8192_bf16", 256, 4, 8192, "bf16", "sbv", 2.0, 0.05,
                                label_smoothing=0.1, reduce_loss=True, seed=1002),
    "c3_bsv32000_bf16_spiked": Workload("c3_bsv32000_bf16_spiked", 2, 512, 32000, "bf16", "bsv",
                                        3.0, 0.10, spike_frac=0.01, seed=1003),
    "c3h_bsv32000_f16_spiked": Workload("c3h_bsv32000_f16_spiked", 1, 2048, 32000, "f16", "bsv",
                                        3.0, 0.10, spike_frac=0.01, seed=1013),
    "c4_bsv65536_bf16_split8": Workload("c4_bsv65536_bf16_split8", 2, 256, 65536, "bf16", "bsv",
                                        2.0, 0.10, label_smoothing=0.1, reduce_loss=True,
                                        seed=1004, vocab_chunks=8),
    "c5_bsv128000_bf16": Workload("c5_bsv128000_bf16", 1, 512, 128000, "bf16", "bsv", 2.0, 0.10,
                                  label_smoothing=0.0, reduce_loss=True, seed=1005),
    "c5_bsv128000_bf16_ls": Workload("c5_bsv128000_bf16_ls", 1, 512, 128000, "bf16", "bsv", 2.0,
                                     0.10, label_smoothing=0.1, reduce_loss=True, seed=1015),
    "c5_bsv128000_f32_ls": Workload("c5_bsv128000_f32_ls", 1, 512, 128000, "f32", "bsv", 2.0,
                                    0.10, label_smoothing=0.1, reduce_loss=True, seed=1025),
    "c5_bsv128000_f32": Workload("c5_bsv128000_f32", 1, 512, 128000, "f32", "bsv", 2.0, 0.10,
                                 label_smoothing=0.0, reduce_loss=True, seed=1035),
    # profiling size of 32 KB rows (the widest the warp path takes): (8, 4096,
    # 16384) bf16, ~1.07 GB
    "c2w_bsv16384_bf16": Workload("c2w_bsv16384_bf16", 8, 4096, 16384, "bf16", "bsv", 2.0, 0.05,
                                  label_smoothing=0.1, reduce_loss=True, seed=1062),
    # profiling size of the 32000-column family: (16, 2048, 32000) bf16, ~2.1 GB
    "c3p_bsv32000_bf16": Workload("c3p_bsv32000_bf16", 16, 2048, 32000, "bf16", "bsv", 3.0,
                                  0.10, spike_frac=0.01, seed=1033),
    # profiling size of the short-row family: (SQ=16384, B=4, 8192) bf16,
    # ~1 GB of logits (several times the L2)
    "c2p_sbv8192_bf16": Workload("c2p_sbv8192_bf16", 16384, 4, 8192, "bf16", "sbv", 2.0, 0.05,
                                 label_smoothing=0.1, reduce_loss=True, seed=1052),
    # profiling size: ~1 GB of bf16 logits (several times the L2)
    "c5p_bsv128000_bf16": Workload("c5p_bsv128000_bf16", 1, 4096, 128000, "bf16", "bsv", 2.0,
                                   0.10, label_smoothing=0.1, reduce_loss=True, seed=1055),
    # profiling size of the widest family: (1, 4096, 256000) bf16, ~2.1 GB
    "c6p_bsv256000_bf16": Workload("c6p_bsv256000_bf16", 1, 4096, 256000, "bf16", "bsv", 2.0,
                                   0.10, label_smoothing=0.1, reduce_loss=True, seed=1066),
    # throughput size: ~4.2 GB of bf16 logits
    "c5t_bsv128000_bf16": Workload("c5t_bsv128000_bf16", 4, 4096, 128000, "bf16", "bsv", 2.0,
                                   0.10, label_smoothing=0.1, reduce_loss=True, seed=1045),
}


def _block_values(w: Workload, b: int) -> np.ndarray:
    r0 = b * ROW_BLOCK
    rows = min(ROW_BLOCK, w.N - r0)
    rng = np.random.default_rng([w.seed, b])
    x = rng.standard_normal((rows, w.V), dtype=np.float32)
    x *= np.float32(w.sigma)
    return x


def spiked_rows(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Rows that get a spike, and the spiked column of each."""
    k = int(np.floor(w.spike_frac * w.N))
    if k == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    rng = np.random.default_rng([w.seed, _SPIKE_STREAM])
    rows = np.sort(rng.permutation(w.N)[:k]).astype(np.int64)
    cols = rng.integers(0, w.V, size=k, dtype=np.int64)
    return rows, cols


def _cast(x32: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(x32).to(DTYPES[dtype])


def logits_rows(w: Workload, r0: int, r1: int) -> torch.Tensor:
    """Rows [r0, r1) of the logits, flattened-row order, as a CPU tensor (rows, V)."""
    out = torch.empty((r1 - r0, w.V), dtype=DTYPES[w.dtype])
    srows, scols = spiked_rows(w)
    b0, b1 = r0 // ROW_BLOCK, (r1 - 1) // ROW_BLOCK
    for b in range(b0, b1 + 1):
        x = _block_values(w, b)
        base = b * ROW_BLOCK
        sel = (srows >= base) & (srows < base + x.shape[0])
        for rr, cc in zip(srows[sel], scols[sel]):
            x[rr - base, cc] += np.float32(w.spike)
        lo, hi = max(r0, base), min(r1, base + x.shape[0])
        out[lo - r0:hi - r0] = _cast(x[lo - base:hi - base], w.dtype)
    return out


def logits(w: Workload, threads: int | None = None, pin_memory: bool = False) -> torch.Tensor:
    """The whole logits tensor, shape (dim0, dim1, V), contiguous, on the CPU."""
    out = torch.empty((w.N, w.V), dtype=DTYPES[w.dtype], pin_memory=pin_memory)
    nblocks = (w.N + ROW_BLOCK - 1) // ROW_BLOCK
    srows, scols = spiked_rows(w)

    def fill(b: int) -> None:
        x = _block_values(w, b)
        base = b * ROW_BLOCK
        sel = (srows >= base) & (srows < base + x.shape[0])
        for rr, cc in zip(srows[sel], scols[sel]):
            x[rr - base, cc] += np.float32(w.spike)
        out[base:base + x.shape[0]] = _cast(x, w.dtype)

    threads = threads or min(16, os.cpu_count() or 1)
    if nblocks == 1 or threads == 1:
        for b in range(nblocks):
            fill(b)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblocks)))
    return out.view(w.dim0, w.dim1, w.V)


def ignored_rows(w: Workload) -> np.ndarray:
    k = int(np.floor(w.ignore_frac * w.N))
    rng = np.random.default_rng([w.seed, _IGNORE_STREAM])
    return np.sort(rng.permutation(w.N)[:k]).astype(np.int64)


def targets(w: Workload) -> torch.Tensor:
    """int64 targets, shape (dim0, dim1), contiguous, on the CPU."""
    rng = np.random.default_rng([w.seed, _TARGET_STREAM])
    t = rng.integers(0, w.V, size=w.N, dtype=np.int64)
    t[ignored_rows(w)] = w.ignore_idx
    return torch.from_numpy(t).view(w.dim0, w.dim1)

