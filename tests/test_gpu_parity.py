"""GPU (through the C ABI) against the CPU oracle on every workload family,
on each path that can run it.  Needs a GB300 and the built library."""
import numpy as np
import pytest
import torch

from tests import harness
from vocabulary_cross_entropy_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

AUTO, ROW, CLUSTER, TWO, STREAM, WARP, VECROW = 0, 1, 2, 3, 4, 5, 6

CASES = [
    ("c1_bsv4096_f32", AUTO, None), ("c1_bsv4096_f32", TWO, None),
    ("c1_bsv4096_f32", STREAM, None), ("c1_bsv4096_f32", ROW, None),
    ("c2_sbv8192_bf16", AUTO, None), ("c2_sbv8192_bf16", CLUSTER, None),
    ("c2_sbv8192_bf16", ROW, None),
    ("c2_sbv8192_bf16", TWO, None), ("c2_sbv8192_bf16", STREAM, None),
    ("c3_bsv32000_bf16_spiked", AUTO, None), ("c3_bsv32000_bf16_spiked", TWO, None),
    ("c3_bsv32000_bf16_spiked", CLUSTER, None),
    ("c3h_bsv32000_f16_spiked", AUTO, None), ("c3h_bsv32000_f16_spiked", TWO, None),
    ("c3h_bsv32000_f16_spiked", CLUSTER, None), ("c1_bsv4096_f32", WARP, None),
    ("c4_bsv65536_bf16_split8", CLUSTER, 8), ("c4_bsv65536_bf16_split8", TWO, 8),
    ("c4_bsv65536_bf16_split8", STREAM, 0), ("c4_bsv65536_bf16_split8", STREAM, 8),
    ("c4_bsv65536_bf16_split8", AUTO, 8), ("c5_bsv128000_bf16_ls", STREAM, 8),
    ("c5_bsv128000_f32_ls", STREAM, 8), ("c2_sbv8192_bf16", STREAM, 3),
    ("c1_bsv4096_f32", STREAM, 5), ("c3h_bsv32000_f16_spiked", STREAM, 16),
    ("c5_bsv128000_bf16", AUTO, None), ("c5_bsv128000_bf16_ls", AUTO, None),
    ("c5_bsv128000_bf16_ls", TWO, None), ("c5_bsv128000_bf16_ls", CLUSTER, None),
    ("c5_bsv128000_f32", AUTO, None), ("c5_bsv128000_f32_ls", AUTO, None),
    ("c5_bsv128000_f32_ls", TWO, None), ("c5_bsv128000_f32_ls", CLUSTER, None),
    ("c1_bsv4096_f32", VECROW, None), ("c2_sbv8192_bf16", VECROW, None),
    ("c3h_bsv32000_f16_spiked", VECROW, None), ("c5_bsv128000_bf16_ls", VECROW, None),
]


@pytest.mark.parametrize("name,path,chunks", CASES,
                         ids=[f"{n}-p{p}" + (f"-k{k}" if k else "") for n, p, k in CASES])
def test_workload_parity(name, path, chunks):
    w = wl.WORKLOADS[name]
    res = harness.run_gpu_vs_oracle(w, force_path=path, num_vocab_chunks=chunks)
    print(name, path, res)


def test_per_row_dloss():
    w = wl.WORKLOADS["c3_bsv32000_bf16_spiked"].with_(dim0=1, dim1=96)
    harness.run_gpu_vs_oracle(w, per_row_dloss=True)
    w = wl.WORKLOADS["c1_bsv4096_f32"].with_(label_smoothing=0.3)
    harness.run_gpu_vs_oracle(w, per_row_dloss=True)


def test_planner_paths():
    import vocabulary_cross_entropy_pass_gb300 as pkg
    dev = torch.device("cuda")
    x = torch.empty(2, 3, 4096, dtype=torch.bfloat16, device=dev)
    assert pkg.ce_plan_path(x)[0] == WARP
    x = torch.empty(2, 3, 128000, dtype=torch.bfloat16, device=dev)
    assert pkg.ce_plan_path(x)[0] == STREAM
    x = torch.empty(2, 3, 4095, dtype=torch.bfloat16, device=dev)  # rows not 16-byte aligned
    assert pkg.ce_plan_path(x)[0] == VECROW
    assert pkg.ce_plan_path(x, pkg.make_options(num_vocab_chunks=2)) == (TWO, 2)
    x = torch.empty(2, 3, 50257, dtype=torch.bfloat16, device=dev)  # wide and off the grid
    assert pkg.ce_plan_path(x) == (STREAM, 1)
    opts = pkg.make_options(force_path=CLUSTER, num_vocab_chunks=8)
    x = torch.empty(2, 256, 65536, dtype=torch.bfloat16, device=dev)
    assert pkg.ce_plan_path(x, opts) == (CLUSTER, 8)
    # a split asked for: the stream kernel with per-chunk partials (chunks of
    # ceil(V/K) rounded up to 16 bytes: 104 bf16 columns in 3 -> 40, 40, 24)
    assert pkg.ce_plan_path(x, pkg.make_options(num_vocab_chunks=8)) == (STREAM, 8)
    x = torch.empty(2, 3, 104, dtype=torch.bfloat16, device=dev)
    assert pkg.ce_plan_path(x, pkg.make_options(num_vocab_chunks=3)) == (STREAM, 3)
    assert pkg.ce_plan_path(x, pkg.make_options(force_path=STREAM, num_vocab_chunks=3)) == (STREAM, 3)
    x = torch.empty(2, 3, 128000, dtype=torch.bfloat16, device=dev)
    assert pkg.ce_plan_path(x, pkg.make_options(num_vocab_chunks=40)) == (TWO, 40)
