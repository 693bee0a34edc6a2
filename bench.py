"""Throughput of the fused vocabulary cross-entropy forward+backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one fused forward+backward pass (ce_fwd_bwd through the C ABI:
ignore-mask count, the main kernel, the fixed-order mean) over the whole
(4, 4096, 128000) bf16 logits batch, label smoothing 0.1, reduce_loss, 10% of
the targets ignored, gradient written in place.  The logits (4.2 GB) are far
larger than the 129 MB L2, so no flush is needed between steps; the in-place
gradient of step k is the input of step k+1 (same bytes, same work).

Prints one JSON line (rank 0).  N > 1 (torchrun, one process per GPU) runs N
independent replicas of the workload (weak scaling, no collective on the data
path); the timed region is bracketed by a barrier and a device synchronize on
every rank and the slowest rank's time is used.

--impl reference times the CPU oracle (oracle/, double precision, OpenMP)
on the host cores, one bounded row block of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CE fwd+bwd tokens/s at V=128000 bf16; achieved HBM GB/s vs GB300 peak"
DEFAULT_WORKLOAD = "c5t_bsv128000_bf16"


def kernels_per_step(path: int, reduce: bool) -> int:
    """The library's launches in one fused step: the count kernel, the main
    kernel (two on the two-stage path), and the mean kernel for a mean on
    the paths that do not take it in their last CTA (stream, warp)."""
    main = 2 if path == 3 else 1
    mean = 1 if reduce and path not in (4, 5) else 0
    return 1 + main + mean


CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


# ----------------------------------------------------------------- byte counts
def logits_bytes(N: int, V: int, elem_bytes: int) -> int:
    return N * V * elem_bytes


def pass_bytes(N: int, V: int, elem_bytes: int) -> int:
    """Algorithmic bytes of one fused pass: read the logits once, write the
    gradient once over them, read the int64 targets."""
    return 2 * logits_bytes(N, V, elem_bytes) + 8 * N


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(w, path: int):
    """DRAM bytes per launch of the main kernel: the reads of the committed
    ncu capture (profiles/ce_stream_kernel_traffic.json), scaled from the
    captured rows to this workload's rows, plus the gradient write the kernel
    must make (every row, ignored ones included: N V s bytes).  A capture's
    own write count misses the dirty lines still in L2 when it ends (~80 MB
    of a 1 GB write), so the write side is the required count, not the
    measured one.  None when the kernel sources changed since the capture, or
    the workload or path differ from what was captured."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ce_stream_kernel_traffic.json")
    if path != 4 or not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    for rel, digest in rec["sources_sha256"].items():
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    from vocabulary_cross_entropy_pass_gb300 import workloads as wl
    cap = wl.WORKLOADS[rec["captured_workload"]]
    if (cap.V, cap.dtype, cap.ignore_frac) != (w.V, w.dtype, w.ignore_frac):
        return None
    return rec["dram_bytes_read"] * w.N / rec["captured_rows"] + logits_bytes(w.N, w.V,
                                                                               w.elem_bytes)


L2_BYTES = 129 * 1000 * 1000  # GB300 L2


def l2_note(logits_bytes: int) -> str:
    """How the timed loop stands to the L2: inputs several times larger than
    it need no flush between steps; smaller ones stay (partly) resident."""
    if logits_bytes >= 4 * L2_BYTES:
        return (f"inputs {logits_bytes / 1e9:.2f} GB >> 129 MB L2 (no flush needed)")
    if logits_bytes > L2_BYTES:
        return (f"inputs {logits_bytes / 1e6:.0f} MB, 1-4x the 129 MB L2 "
                "(not flushed: partly L2-resident)")
    return f"inputs {logits_bytes / 1e6:.1f} MB, smaller than the 129 MB L2 (L2-resident)"


def aggregate(local_ms: float, local_tokens: int, world: int, all_reduce_max=None):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time.  all_reduce_max(x) returns the max of x over ranks."""
    ms = all_reduce_max(local_ms) if all_reduce_max else local_ms
    return ms, local_tokens * world / (ms / 1e3)


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons, stamped with
    host time so the samples inside the timed region can be picked out."""

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms), "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(CLOCK_FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = len(inside)
        if not inside and self.samples:
            # region shorter than the sampling period: nearest samples around it
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for (_, p) in near]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(p[0]) for p in inside) if v is not None)
        smax = max((v for v in (num(p[1]) for p in inside) if v is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in inside for k in range(4) if p[4 + k] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(inside), "window_samples": window,
                "power_w_max": max((v for v in (num(p[2]) for p in inside) if v is not None),
                                   default=None)}


# ----------------------------------------------------------------- CPU oracle timing
_ORACLE_CODE = {"f32": 0, "bf16": 1, "f16": 2}


def _storage(x):
    """Raw storage of a CPU tensor as numpy (float32, or uint16 bit patterns)."""
    import numpy as np
    import torch
    x = x.contiguous()
    if x.dtype == torch.float32:
        return x.numpy().ravel()
    return x.view(torch.int16).numpy().view(np.uint16).ravel()


def oracle_rows_per_s(w, x_host, t_host, budget_s: float, block: int = 256, max_rows=None):
    """Time the CPU oracle (fwd+bwd, double) on consecutive row blocks of the
    workload until `budget_s` seconds have passed.  Returns (rows/s, rows,
    seconds, threads)."""
    import numpy as np

    import oracle
    lib = oracle.load()
    rows_done, t_used = 0, 0.0
    r0 = 0
    x2 = x_host.view(w.N, w.V)
    t1d = t_host.reshape(-1)
    limit = w.N if max_rows is None else min(w.N, max_rows)
    while t_used < budget_s and rows_done < limit:
        r1 = min(limit, r0 + block)
        xs = _storage(x2[r0:r1])
        ts = t1d[r0:r1].numpy()
        t = time.perf_counter()
        oracle.ce(xs, _ORACLE_CODE[w.dtype], 1, r1 - r0, w.V, targets=ts,
                  label_smoothing=w.label_smoothing, reduce_loss=True,
                  dloss=np.array([1.0]), lib=lib)
        t_used += time.perf_counter() - t
        rows_done += r1 - r0
        r0 = r1 % limit
    return rows_done / t_used, rows_done, t_used, oracle.num_threads(lib)


def torch_cross_entropy(w, x, t, steps: int = 5, warmup: int = 3) -> dict:
    """PyTorch's own cross-entropy on the same device logits, for context:
    F.cross_entropy (mean, ignore_index, label_smoothing) and its autograd
    backward per step, timed with CUDA events on the current stream."""
    import torch
    import torch.nn.functional as F
    xr = x.view(w.N, w.V).detach().requires_grad_(True)
    tr = t.reshape(-1)

    def step():
        loss = F.cross_entropy(xr, tr, ignore_index=w.ignore_idx,
                               label_smoothing=w.label_smoothing,
                               reduction="mean" if w.reduce_loss else "none")
        (loss if w.reduce_loss else loss.sum()).backward()
        xr.grad = None

    for _ in range(warmup):
        step()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record()
    for _ in range(steps):
        step()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / steps
    return {"value": w.N / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "what": "torch.nn.functional.cross_entropy forward + autograd backward (eager, "
                    f"torch {torch.__version__}) on the same device logits"}


# ----------------------------------------------------------------- arms
def run_reference(args, w, rank: int, world: int) -> None:
    if rank != 0:
        return
    import numpy as np

    import oracle
    from vocabulary_cross_entropy_pass_gb300 import workloads as wl
    lib = oracle.load()
    R = args.ref_rows
    nblk = (w.N + R - 1) // R
    t_all = wl.targets(w).view(-1)
    # a few row blocks spread over the workload, generated once; the steps
    # take them in turn (the oracle's speed does not depend on which rows)
    picks = sorted({(k * nblk) // 4 for k in range(4)})
    blocks = []
    for b in picks:
        r0, r1 = b * R, min(w.N, (b + 1) * R)
        blocks.append((_storage(wl.logits_rows(w, r0, r1)), t_all[r0:r1].numpy(), r1 - r0))

    def step(i):
        xs, ts, rows = blocks[i % len(blocks)]
        t = time.perf_counter()
        oracle.ce(xs, _ORACLE_CODE[w.dtype], 1, rows, w.V, targets=ts,
                  label_smoothing=w.label_smoothing, reduce_loss=True, dloss=np.array([1.0]),
                  lib=lib)
        return time.perf_counter() - t, rows

    for i in range(args.warmup):
        step(i)
    tot_t, tot_rows = 0.0, 0
    for i in range(args.steps):
        dt, rows = step(args.warmup + i)
        tot_t += dt
        tot_rows += rows
    value = tot_rows / tot_t
    cores = oracle.num_threads(lib)
    sample = (f"{R} rows of the workload per step ({len(blocks)} row blocks spread over it, "
              "in turn), fwd+bwd in double")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, args) -> dict:
    return {"workload": f"{w.name}: logits ({w.dim0},{w.dim1},{w.V}) {w.dtype} "
                        f"({'B,SQ,V' if w.layout == 'bsv' else 'SQ,B,V'}), N={w.N} rows, "
                        f"sigma={w.sigma}, {int(w.ignore_frac * 100)}% ignored, "
                        f"label_smoothing={w.label_smoothing}, reduce_loss={w.reduce_loss}, "
                        "gradient in place",
            "tokens_per_step": w.N, "vocab": w.V, "logits_dtype": w.dtype,
            "accumulate": "f32", "l2": l2_note(w.logits_bytes),
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def run_ours(args, w, rank: int, world: int, dist) -> None:
    import torch

    import vocabulary_cross_entropy_pass_gb300 as pkg
    from vocabulary_cross_entropy_pass_gb300 import workloads as wl

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    # inputs: pinned host copy (also the e2e source) and a resident device copy
    x_host = wl.logits(w, pin_memory=True)
    t_host = wl.targets(w).pin_memory()
    x = x_host.to(dev, non_blocking=True)
    t = t_host.to(dev, non_blocking=True)
    # one mean, or one loss per row
    loss = torch.empty(1 if w.reduce_loss else w.N, dtype=torch.float32, device=dev)
    tune = dict(force_path=args.force_path, num_vocab_chunks=args.chunks,
                tune_threads=args.tune_threads, tune_stages=args.tune_stages,
                tune_ctas_per_sm=args.tune_ctas_per_sm, tune_l2_keep=args.tune_l2_keep,
                tune_tile_kb=args.tune_tile_kb)
    opts = pkg.make_options(**tune)
    ws = torch.empty(pkg.ce_workspace_bytes(w.dim0, w.dim1, w.V, x.dtype, opts),
                     dtype=torch.uint8, device=dev)
    path, chunks = pkg.ce_plan_path(x, opts)
    torch.cuda.synchronize(dev)

    mode = args.mode
    if mode == "fused":
        def step(o=opts):
            pkg.ce_fwd_bwd(x, t, label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                           reduce_loss=w.reduce_loss, loss_out=loss, workspace=ws, opts=o)
    elif mode == "weighted":
        # per-class weights (torch F.cross_entropy(weight=...)): the stream kernel
        # when rows and weights are aligned, else the two-stage kernels
        cw = torch.empty(w.V, dtype=torch.float32, device=dev).uniform_(0.1, 3.0)

        def step(o=opts):
            pkg.ce_fwd_bwd(x, t, label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                           reduce_loss=w.reduce_loss, loss_out=loss, workspace=ws, opts=o,
                           class_weights=cw)
    elif mode == "linear":
        # lm_head (hidden . W^T) + cross-entropy + both gradients, chunked over rows
        del x
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed)
        hid = (torch.randn(w.N, args.hidden, device=dev, generator=gen)).to(torch.bfloat16)
        wmat = (torch.randn(w.V, args.hidden, device=dev, generator=gen)
                / args.hidden ** 0.5 * 2).to(torch.bfloat16)
        gh = torch.empty_like(hid)
        gw = torch.zeros(w.V, args.hidden, dtype=torch.float32, device=dev)
        lws = torch.empty(pkg._lib.load().ce_linear_workspace_bytes(
            w.N, args.hidden, w.V, 1, args.chunk_rows), dtype=torch.uint8, device=dev)
        t_flat = t.reshape(-1)

        def step(o=opts):
            pkg.ce_linear_fwd_bwd(hid, wmat, t_flat, label_smoothing=w.label_smoothing,
                                  ignore_idx=w.ignore_idx, reduce_loss=w.reduce_loss,
                                  grad_hidden=gh, grad_weight=gw, chunk_rows=args.chunk_rows,
                                  loss_out=loss, workspace=lws)
    elif mode == "split":
        # forward only (saves lse and the kept-row count), then the backward
        lse = torch.empty(w.N, dtype=torch.float32, device=dev)
        n_kept = torch.empty(1, dtype=torch.int64, device=dev)

        def step(o=opts):
            pkg.ce_fwd_only(x, t, label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                            reduce_loss=w.reduce_loss, loss_out=loss, lse_out=lse,
                            n_non_ignore_out=n_kept, workspace=ws, opts=o)
            pkg.ce_bwd(x, t, lse, label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                       reduce_loss=w.reduce_loss, n_non_ignore=n_kept, grad=x)
    else:
        # vocabulary shards held as separate tensors, the three steps per pass
        R = args.vocab_shards
        c = -(-w.V // R)
        shards = [x[..., k * c:min(w.V, (k + 1) * c)].contiguous() for k in range(R)]
        del x
        offsets = [min(w.V, k * c) for k in range(R)] + [w.V]
        part = torch.empty(R, w.N, 4, dtype=torch.float32, device=dev)
        lse = torch.empty(w.N, dtype=torch.float32, device=dev)
        n_kept = torch.empty(1, dtype=torch.int64, device=dev)

        def step(o=opts):
            for k, sh in enumerate(shards):
                pkg.ce_vp_partials(sh, t, offsets[k], partials=part[k], ignore_idx=w.ignore_idx)
            pkg.ce_vp_combine(part, offsets, t, label_smoothing=w.label_smoothing,
                              ignore_idx=w.ignore_idx, reduce_loss=w.reduce_loss, loss_out=loss,
                              lse_out=lse, n_non_ignore_out=n_kept, workspace=ws)
            for k, sh in enumerate(shards):
                pkg.ce_vp_bwd(sh, t, offsets[k], w.V, lse, label_smoothing=w.label_smoothing,
                              ignore_idx=w.ignore_idx, reduce_loss=w.reduce_loss,
                              n_non_ignore=n_kept, grad=sh)

    for _ in range(args.warmup):
        step()
    st, err = pkg.ce_get_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {err:#x} after warm-up")

    # per-launch events around the main kernel, on the launching stream
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for (b, e) in evs:  # torch creates an event on its first record
        b.record(stream)
        e.record(stream)
    torch.cuda.synchronize(dev)
    step_opts = [pkg.make_options(event_begin=b.cuda_event, event_end=e.cuda_event, **tune)
                 for (b, e) in evs]
    assert all(o.event_begin and o.event_end for o in step_opts)

    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    # The main kernel's own duration (the roofline's time) from a second run
    # of the same steps with events recorded around it.  An event recorded
    # between the count kernel and the main kernel keeps the main kernel from
    # starting under the count kernel (programmatic dependent launch), so the
    # steps above, whose time is the headline, carry none.
    torch.cuda.synchronize(dev)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for i in range(args.steps):
        step(step_opts[i])
    k1.record(stream)
    torch.cuda.synchronize(dev)
    t2 = time.time()
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    clocks_kernel_run = sampler.summary(t1, t2)
    total_ms = start.elapsed_time(end)
    kernel_run_ms = k0.elapsed_time(k1) / args.steps
    kernel_ms = (sum(b.elapsed_time(e) for (b, e) in evs) / args.steps
                 if args.mode in ("fused", "split") else None)

    def allmax(v):
        if dist is None:
            return v
        tt = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())

    ms, tok_s = aggregate(total_ms, w.N * args.steps, world, allmax)

    if mode == "linear":
        # tensor-bound: three GEMMs of 2 N V H flops each per step
        if rank == 0:
            flops = 6.0 * w.N * w.V * args.hidden
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                pk = json.load(f)
            peak = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops", 1700.0)))
            ach = flops / (ms / args.steps / 1e3) / 1e12
            line = {"metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "bf16", "data": "synthetic",
                    "config": config_of(w, args) | {"mode": "linear", "hidden": args.hidden,
                                                     "chunk_rows": args.chunk_rows,
                                                     "logits_gemm": args.linear_gemm},
                    "roofline": {"bound": "tensor", "kernel": "whole step (3 GEMMs + CE)",
                                 "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                                 "frac": ach / peak, "traffic": None,
                                 "peak_source": "measured bf16_tflops_sustained"},
                    "clocks": clocks}
            print(json.dumps(line), flush=True)
        return
    if mode != "fused":
        # one line for a secondary mode: whole-step bytes over whole-step time
        if rank == 0:
            # logits passes through HBM: the stream and warp kernels read once
            # and write once, the split, two-stage and vocabulary-parallel
            # steps read twice
            passes = 3
            if mode == "weighted":
                wopts = pkg.make_options(**tune)
                wopts.class_weights = cw.data_ptr()
                if pkg.ce_plan_path(x, opts=wopts)[0] in (pkg.CE_PATH_STREAM, pkg.CE_PATH_WARP):
                    passes = 2
            nb = passes * w.logits_bytes + 8 * w.N
            line = {"metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f32", "data": "synthetic",
                    "config": config_of(w, args) | {"mode": mode,
                                                     "vocab_shards": args.vocab_shards
                                                     if mode == "vp" else None},
                    "roofline": {"bound": "hbm",
                                 "kernel": f"whole step ({passes - 1} reads + one write)",
                                 "note": "weighted mode: the class weights are read from L2"
                                 if mode == "weighted" else None,
                                 "achieved": nb / (ms / args.steps / 1e3) / 1e9,
                                 "peak": measured_peaks()["hbm_gbs"], "unit": "GB/s",
                                 "frac": nb / (ms / args.steps / 1e3) / 1e9
                                 / measured_peaks()["hbm_gbs"], "traffic": None},
                    "clocks": clocks}
            print(json.dumps(line), flush=True)
        return

    # end to end through the public call: every step copies its inputs from
    # pinned host memory to the device, runs the pass and reads the loss back.
    # Two device input buffers let the copy of step k+1 (copy stream) overlap
    # the pass of step k (compute stream); each buffer is refilled only after
    # the pass that used it has finished.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    h2d = w.logits_bytes + 8 * w.N
    xs = [x, torch.empty_like(x)]
    ts_ = [t, torch.empty_like(t)]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    loss_host = torch.empty(max(e2e_steps, 2), loss.numel(), dtype=torch.float32, pin_memory=True)

    def e2e_round(k):
        b = k % 2
        copy_stream.wait_event(done[b])
        with torch.cuda.stream(copy_stream):
            xs[b].copy_(x_host, non_blocking=True)
            ts_[b].copy_(t_host, non_blocking=True)
            copied[b].record(copy_stream)
        stream.wait_event(copied[b])
        pkg.ce_fwd_bwd(xs[b], ts_[b], label_smoothing=w.label_smoothing, ignore_idx=w.ignore_idx,
                       reduce_loss=w.reduce_loss, loss_out=loss, workspace=ws, opts=opts,
                       stream=stream)
        loss_host[k].copy_(loss, non_blocking=True)
        done[b].record(stream)

    # warm-up: the first write into a freshly allocated device buffer and the
    # first copy on the copy stream carry one-time costs
    for ev in done:
        ev.record(stream)
    for k in range(2):
        e2e_round(k)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for ev in done:
        ev.record(stream)
    for k in range(e2e_steps):
        e2e_round(k)
    e2.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, e2e_tok_s = aggregate(s2.elapsed_time(e2), w.N * e2e_steps, world, allmax)
    st, err = pkg.ce_get_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {err:#x}")
    if rank != 0:
        return

    peaks = measured_peaks()
    nbytes = pass_bytes(w.N, w.V, w.elem_bytes)
    traffic = profiled_traffic(w, path)
    torch_ref = None if args.no_torch_ref else torch_cross_entropy(w, x, t)
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        rps, rows, secs, cores = oracle_rows_per_s(w, x_host, t_host, args.cpu_budget)
        cpu = {"value": rps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} rows of the workload in row blocks of 256 "
                         f"({secs:.1f} s of oracle time, fwd+bwd in double)"}
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, see vocabulary_cross_entropy_pass_gb300/workloads.py)",
        "config": config_of(w, args) | {"path": {1: "row", 2: "cluster", 3: "two_stage", 4: "stream",
                                                 5: "warp", 6: "vecrow"}[path],
                                         "vocab_chunks": chunks},
        "hbm_gbs_formula": nbytes * args.steps * world / (ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic,
                     "traffic_source": "ncu dram__bytes_read of the committed capture "
                                       "(profiles/ce_stream_kernel_traffic.json) scaled by "
                                       "rows + the required gradient write N*V*s",
                     "achieved_is": "algorithmic bytes (logits read + "
                                    "gradient write + targets) / kernel time",
                     "dram_gbs": traffic / (kernel_ms / 1e3) / 1e9 if traffic else None,
                     "dram_frac": traffic / (kernel_ms / 1e3) / 1e9 / peaks["hbm_gbs"]
                     if traffic else None,
                     "peak_source": peaks["source"], "kernel_ms": kernel_ms,
                     "kernel_ms_how": "CUDA events around the main kernel on the launching "
                                      "stream, over a second run of the timed steps (its "
                                      f"steps took {kernel_run_ms:.4f} ms each; SM clock "
                                      f"median {clocks_kernel_run.get('sm_mhz')} MHz)",
                     "algorithmic_bytes": nbytes},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_tok_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4 * loss.numel(), "steps": e2e_steps,
                "ms_per_step": e2e_ms / e2e_steps,
                "how": "ce_fwd_bwd per step on inputs copied from pinned host memory "
                       "(two device buffers: the copy of step k+1 overlaps the pass of "
                       "step k) and the loss read back"},
        "gpu_launches": kernels_per_step(path, w.reduce_loss) * args.steps,
        "torch_cross_entropy": torch_ref,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-torch-ref", action="store_true")
    # secondary passes: "split" = ce_fwd_only + ce_bwd (autograd order), "vp" = the
    # vocabulary-parallel steps over --vocab-shards shards on one GPU, "weighted" =
    # the class-weighted pass, "linear" = lm_head + cross-entropy chunked over rows
    ap.add_argument("--mode", choices=["fused", "split", "vp", "weighted", "linear"],
                    default="fused")
    ap.add_argument("--hidden", type=int, default=4096)      # linear mode: H
    ap.add_argument("--chunk-rows", type=int, default=4096)  # linear mode: rows per chunk
    # linear mode: "library" puts the logits GEMM on cuBLAS (GBCE_LINEAR_GEMM)
    ap.add_argument("--linear-gemm", choices=["tcgen05", "library"], default="tcgen05")
    ap.add_argument("--vocab-shards", type=int, default=8)
    # planner overrides, for tuning sweeps (defaults: the planner's choice)
    ap.add_argument("--force-path", type=int, default=0)
    ap.add_argument("--chunks", type=int, default=0)
    ap.add_argument("--tune-threads", type=int, default=0)
    ap.add_argument("--tune-stages", type=int, default=0)
    ap.add_argument("--tune-ctas-per-sm", type=int, default=0)
    ap.add_argument("--tune-l2-keep", type=int, default=0)
    ap.add_argument("--tune-tile-kb", type=int, default=0)
    # another vocabulary width and/or row count for the chosen workload (its
    # dtype, value spread, ignore fraction and smoothing kept), as (1, rows, V)
    ap.add_argument("--vocab", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.vocab < 0 or args.rows < 0:
        ap.error("--vocab and --rows must be positive")

    from vocabulary_cross_entropy_pass_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    if args.vocab or args.rows:
        V = args.vocab or w.V
        N = args.rows or w.N
        w = w.with_(name=f"{w.name}_as_{N}x{V}", dim0=1, dim1=N, V=V, layout="bsv",
                    vocab_chunks=0)
    if args.linear_gemm == "library":
        os.environ["GBCE_LINEAR_GEMM"] = "library"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return 0
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
