"""Host logic of bench.py on the CPU: byte counts, the whole-job aggregate over
ranks (world size 2, gloo), the reference arm's JSON line, clock summaries."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_pass_bytes_throughput_workload():
    # (4, 4096, 128000) bf16: 4,194,304,000 B of logits read and written + int64 targets
    assert bench.pass_bytes(16384, 128000, 2) == 8_388_739_072


def test_kernels_per_step():
    # count kernel + main kernel(s) + the mean kernel where the path does not
    # take the mean in its last CTA
    assert bench.kernels_per_step(4, True) == 2   # stream
    assert bench.kernels_per_step(5, True) == 2   # warp
    assert bench.kernels_per_step(3, True) == 4   # two-stage: two kernels + mean
    assert bench.kernels_per_step(3, False) == 3
    assert bench.kernels_per_step(6, True) == 3   # plain-load rows
    assert bench.kernels_per_step(6, False) == 2
    assert bench.kernels_per_step(1, False) == 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def allmax(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    local_ms = 100.0 + 50.0 * rank       # rank 1 is the slow one
    ms, tok_s = bench.aggregate(local_ms, 1000, world, allmax)
    out[rank] = (ms, tok_s)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for r in (0, 1):
        ms, tok_s = out[r]
        assert ms == 150.0                       # the slowest rank's time
        assert tok_s == pytest.approx(2 * 1000 / 0.150)


def test_reference_arm_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--workload", "c1_bsv4096_f32", "--ref-rows", "8"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--workload", "c1_bsv4096_f32"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_clock_summary_flags_throttling():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(1.0, ["1900", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active",
                        "Not Active"]),
                 (1.1, ["1800", "2070", "950", "0x4", "Not Active", "Not Active", "Not Active",
                        "Active"]),
                 (1.2, ["2000", "2070", "980", "0x0", "Not Active", "Not Active", "Not Active",
                        "Not Active"])]
    c = s.summary(0.9, 1.3)
    assert c["sm_mhz"] == 1900.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The committed ncu record counts only while the kernel sources it names
    are unchanged; it is scaled by rows to the bench workload."""
    import hashlib
    import shutil
    from vocabulary_cross_entropy_pass_gb300 import workloads as wl
    w = wl.WORKLOADS["c5t_bsv128000_bf16"]
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "vocabulary_cross_entropy_pass_gb300" / "csrc"
    csrc.mkdir(parents=True)
    digests = {}
    for f in ("ce_stream.cu", "ce_device.cuh"):
        src = os.path.join(ROOT, "vocabulary_cross_entropy_pass_gb300", "csrc", f)
        shutil.copy(src, csrc / f)
        digests[f"vocabulary_cross_entropy_pass_gb300/csrc/{f}"] = hashlib.sha256(
            open(src, "rb").read()).hexdigest()
    rec = json.load(open(os.path.join(ROOT, "profiles", "ce_stream_kernel_traffic.json")))
    rec["sources_sha256"] = digests
    json.dump(rec, open(root / "profiles" / "ce_stream_kernel_traffic.json", "w"))
    monkeypatch.setattr(bench, "ROOT", str(root))
    t = bench.profiled_traffic(w, 4)
    # the capture covers rec["captured_rows"] rows; the bench workload has
    # 16384: its reads scale by rows, the write is the gradient of every row
    write = w.N * w.V * 2
    assert t == rec["dram_bytes_read"] * w.N / rec["captured_rows"] + write
    # the kernel skips the reads of ignored rows (10 %) and no more: the
    # traffic lies between the required read + write and the formula bytes
    kept_read = (w.N - int(w.ignore_frac * w.N)) * w.V * 2
    assert kept_read + write <= t < 1.02 * bench.pass_bytes(w.N, w.V, 2)
    assert bench.profiled_traffic(w, 2) is None          # another path: no counters
    assert bench.profiled_traffic(w.with_(V=64000), 4) is None
    with open(csrc / "ce_stream.cu", "a") as f:          # a changed kernel voids them
        f.write("\n// edited\n")
    assert bench.profiled_traffic(w, 4) is None
