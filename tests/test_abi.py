"""The C ABI on the CPU: the library loads, exports every function the header
declares, sizes workspaces, and rejects bad arguments on the host before any
CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from vocabulary_cross_entropy_pass_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ce.h")


@pytest.fixture(scope="module")
def lib():
    from vocabulary_cross_entropy_pass_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(ce_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_known_entry_points():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # exported with C linkage: no mangled names needed
    nm = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", nm, flags=re.M), name


def test_status_strings(lib):
    for code in range(9):
        s = lib.ce_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ce_status_string(99).decode() == "unknown status"


def test_workspace_bytes(lib):
    ws = lib.ce_workspace_bytes(4, 4096, 128000, 1, None)
    # header + per-row losses + per-(row, chunk) partials of the fallback path
    # (chunks of up to 16384 columns: 8 for V = 128000)
    assert ws >= 256 + 4 * 16384 + 16 * 16384 * 8
    assert lib.ce_workspace_bytes(-1, 4, 10, 1, None) == 0
    assert lib.ce_workspace_bytes(1, 4, 0, 1, None) == 0
    assert lib.ce_workspace_bytes(1, 4, 10, 7, None) == 0
    o = _lib.make_options(num_vocab_chunks=8)
    assert lib.ce_workspace_bytes(2, 256, 65536, 1, ctypes.byref(o)) >= 16 * 512 * 8


def _call(lib, **kw):
    args = dict(logits=0x1000, dtype=1, layout=0, d0=2, d1=3, V=4096, strides=(3 * 4096, 4096, 1),
                targets=0x2000, tstrides=(3, 1), a=0.0, ignore=-100, reduce=0, dloss=None,
                loss=0x3000, grad=None, n=None, ws=0x4000, wsb=1 << 30, opts=None)
    args.update(kw)
    if args["grad"] is None:
        args["grad"] = args["logits"]
    return lib.ce_fwd_bwd(ctypes.c_void_p(args["logits"]), args["dtype"], args["layout"], args["d0"],
                          args["d1"], args["V"], _lib.i64_array(args["strides"]),
                          ctypes.c_void_p(args["targets"]), _lib.i64_array(args["tstrides"]),
                          args["a"], args["ignore"], args["reduce"], ctypes.c_void_p(args["dloss"]),
                          ctypes.c_void_p(args["loss"]), ctypes.c_void_p(args["grad"]),
                          ctypes.c_void_p(args["n"]), ctypes.c_void_p(args["ws"]), args["wsb"],
                          args["opts"], None)


def test_host_validation_rejects_before_launch(lib):
    # every case below fails in the host checks, before any CUDA call
    assert _call(lib, dtype=5) == 2
    assert _call(lib, layout=2) == 1
    assert _call(lib, logits=0) == 1
    assert _call(lib, targets=0) == 1
    assert _call(lib, loss=0) == 1
    assert _call(lib, ws=0) == 1
    assert _call(lib, V=0) == 1
    assert _call(lib, d0=-1) == 1
    assert _call(lib, a=1.5) == 1
    assert _call(lib, a=float("nan")) == 1
    assert _call(lib, strides=(3 * 4096, 4096, 2)) == 3
    assert _call(lib, strides=(-1, 4096, 1)) == 3
    assert _call(lib, tstrides=(-3, 1)) == 3
    assert _call(lib, ws=0x4008) == 1          # not 16-byte aligned
    assert _call(lib, logits=0x1001) == 1      # bf16 logits off a 2-byte boundary
    assert _call(lib, logits=0x1002, dtype=0) == 1  # fp32 logits off a 4-byte boundary
    assert _call(lib, wsb=100) == 4
    assert _call(lib, grad=0x9000) == 1        # the gradient must go in place
    o = _lib.make_options()
    o.reserved[1] = 1
    assert _call(lib, opts=ctypes.byref(o)) == 1
    o = _lib.make_options(tune_threads=300)
    assert _call(lib, opts=ctypes.byref(o)) == 1
    o = _lib.make_options(tune_l2_keep=3)
    assert _call(lib, opts=ctypes.byref(o)) == 1
    o = _lib.make_options(force_path=7)
    assert _call(lib, opts=ctypes.byref(o)) == 1


def test_planner(lib):
    def plan(V, dtype=1, strides=None, base=0x1000, **o):
        opts = _lib.make_options(**o)
        ch = ctypes.c_int(0)
        st = strides or (3 * V, V, 1)
        p = lib.ce_plan_path(ctypes.c_void_p(base), dtype, 2, 3, V, _lib.i64_array(st),
                             ctypes.byref(opts), ctypes.byref(ch))
        return p, ch.value
    assert plan(4096) == (5, 1)                    # a row fits one 16 KB tile: warp path
    assert plan(8192) == (5, 1)
    assert plan(16384) == (5, 1)                   # 32 KB tile
    assert plan(16392) == (4, 1)                   # wider than a tile: stream path
    assert plan(4096, force_path=1) == (1, 1)      # the fused row kernel on request
    assert plan(16392, force_path=5)[0] == -2
    assert plan(32000) == (4, 1)                   # wider than one CTA: stream path
    assert plan(128000) == (4, 1)
    assert plan(128000, dtype=0) == (4, 1)
    assert plan(128000, force_path=2) == (2, 16)
    assert plan(32000, force_path=2) == (2, 4)
    assert plan(4096, force_path=4) == (4, 1)
    assert plan(4095, force_path=4) == (4, 1)      # rows off the grid: TMA body, scalar edges
    assert plan(4095, force_path=5)[0] == -2       # the warp path needs aligned rows
    assert plan(65536, num_vocab_chunks=8, force_path=2) == (2, 8)
    assert plan(65536, num_vocab_chunks=8, force_path=3) == (3, 8)
    assert plan(4095) == (6, 1)                    # rows not 16-byte aligned: plain loads
    assert plan(4096, base=0x1002) == (6, 1)       # base not 16-byte aligned
    assert plan(100277) == (4, 1)                  # ... over 32 KB: the stream kernel
    assert plan(32000, base=0x1002) == (4, 1)
    assert plan(100277, tune_threads=512) == (6, 1)  # a shape only the plain-load kernel has
    assert plan(100277, force_path=4, tune_threads=512)[0] == -2
    # a vocabulary split asked for: the stream kernel combines up to 32 chunk
    # partials (chunks of ceil(V/K) rounded up to 16 bytes), the two-stage
    # kernels more; the cluster kernel on request
    assert plan(65536, num_vocab_chunks=8) == (4, 8)
    assert plan(65536, num_vocab_chunks=8, force_path=4) == (4, 8)
    assert plan(128000, num_vocab_chunks=8) == (4, 8)
    assert plan(104, num_vocab_chunks=3) == (4, 3)
    assert plan(104, num_vocab_chunks=3, force_path=4) == (4, 3)  # chunks of 40, 40, 24
    assert plan(16, num_vocab_chunks=8, force_path=4) == (4, 2)   # 8 columns each: two
    assert plan(128000, num_vocab_chunks=32) == (4, 32)           # 8000-byte chunks
    assert plan(128000, num_vocab_chunks=32, force_path=4) == (4, 32)
    assert plan(128000, num_vocab_chunks=40) == (3, 40)
    assert plan(128000, num_vocab_chunks=40, force_path=4)[0] == -2
    assert plan(4095, num_vocab_chunks=4, force_path=4)[0] == -2
    assert plan(4096, force_path=6) == (6, 1)      # aligned rows on request
    assert plan(4095, num_vocab_chunks=4) == (3, 4)  # a split asked for: two-stage
    assert plan(4095, force_path=3) == (3, 1)
    assert plan(4095, force_path=6, num_vocab_chunks=2)[0] == -2
    assert plan(4095, tune_threads=1024) == (6, 1)  # the plain-load kernel's other shapes
    assert plan(4095, tune_threads=32) == (6, 1)
    assert plan(128000, tune_threads=1024)[0] == -2  # the stream kernel has no such shape
    assert plan(4096, force_path=1, tune_threads=32)[0] == -2
    assert plan(4096, force_path=1, base=0x1002)[0] == -2
    assert plan(4_000_000)[0] == 4                 # any width streams
    assert plan(4_000_000, force_path=2)[0] == -2  # too wide for 16 CTAs
    assert plan(32000, force_path=1)[0] == -2      # one CTA cannot hold the row
    assert plan(4096, force_path=2) == (2, 2)
    # class weights: the stream kernel when rows and weights are 16-byte
    # aligned (any width), else the two-stage kernels; paths without weights
    # are refused; a ring too shallow for a 16-bit tile and its two weight
    # slots twice falls back to two-stage (fp32 tiles need one weight slot)
    assert plan(128000, class_weights=0x2000)[0] == 4
    assert plan(4096, class_weights=0x2000)[0] == 4
    assert plan(128000, class_weights=0x2004)[0] == 3
    assert plan(4095, class_weights=0x2000)[0] == 3
    assert plan(4096, class_weights=0x2000, force_path=5)[0] == -2
    assert plan(4096, class_weights=0x2000, force_path=1)[0] == -2
    assert plan(128000, class_weights=0x2000, tune_stages=4)[0] == 3
    assert plan(128000, dtype=0, class_weights=0x2000, tune_stages=4)[0] == 4
    assert plan(128000, class_weights=0x2000, num_vocab_chunks=4)[0] == 3


def test_overlapping_rows_rejected_for_in_place_gradient(lib):
    # a broadcast (stride 0) or rows closer than V apart cannot take an in-place gradient
    assert _call(lib, strides=(0, 4096, 1)) == 3
    assert _call(lib, strides=(3 * 4096, 100, 1)) == 3
    # a transposed (SQ, B, V) storage read as (B, SQ, V) passes the host checks
    # and fails later only for want of a GPU
    assert _call(lib, d0=2, d1=3, strides=(4096, 2 * 4096, 1)) not in (1, 2, 3, 4)


def test_error_getters_reject_null_pointers(lib):
    # no CUDA call is made before these checks
    err = ctypes.c_uint32(0)
    assert lib.ce_get_error(None, None, ctypes.byref(err)) == 1
    assert lib.ce_get_error(ctypes.c_void_p(0x1000), None, None) == 1
    assert lib.ce_noalloc_get_error(None, None) == 1


def test_bwd_host_validation(lib):
    def call(**kw):
        a = dict(logits=0x1000, dtype=1, d0=2, d1=3, V=4096, st=(3 * 4096, 4096, 1), tgt=0x2000,
                 ts=(3, 1), lse=0x3000, a=0.0, reduce=0, dloss=None, n=None, grad=0x9000,
                 gst=(3 * 4096, 4096, 1))
        a.update(kw)
        return lib.ce_bwd(ctypes.c_void_p(a["logits"]), a["dtype"], 0, a["d0"], a["d1"], a["V"],
                          _lib.i64_array(a["st"]), ctypes.c_void_p(a["tgt"]),
                          _lib.i64_array(a["ts"]), ctypes.c_void_p(a["lse"]), a["a"], -100,
                          a["reduce"], ctypes.c_void_p(a["dloss"]), ctypes.c_void_p(a["n"]),
                          ctypes.c_void_p(a["grad"]), _lib.i64_array(a["gst"]), None)
    assert call(lse=0) == 1
    assert call(grad=0) == 1
    assert call(reduce=1) == 1                       # the mean needs the forward's count
    assert call(gst=(3 * 4096, 4096, 2)) == 3
    assert call(gst=(0, 4096, 1)) == 3               # gradient rows may not share memory
    assert call(grad=0x1000, gst=(4096, 2 * 4096, 1)) == 3  # in place means the same strides
    assert call(dtype=9) == 2
    assert call(logits=0x1001) == 1                   # off the element size
    assert call(grad=0x9001) == 1
    assert call(d0=0) == 0                            # nothing to do


def test_vocab_parallel_host_validation(lib):
    def comb(offs, R=None, **kw):
        R = len(offs) - 1 if R is None else R
        a = dict(part=0x1000, d0=1, d1=4, tgt=0x2000, ts=(4, 1), a=0.0, reduce=0, loss=0x3000,
                 lse=0x4000, n=None, ws=0x5000, wsb=1 << 20)
        a.update(kw)
        return lib.ce_vp_combine(ctypes.c_void_p(a["part"]), R, _lib.i64_array(offs), a["d0"],
                                 a["d1"], ctypes.c_void_p(a["tgt"]), _lib.i64_array(a["ts"]),
                                 a["a"], -100, a["reduce"], ctypes.c_void_p(a["loss"]),
                                 ctypes.c_void_p(a["lse"]), ctypes.c_void_p(a["n"]),
                                 ctypes.c_void_p(a["ws"]), a["wsb"], None)
    assert comb([0, 10, 10, 30]) == 1          # empty shard: offsets must increase
    assert comb([1, 10, 30]) == 1              # must start at column 0
    assert comb(list(range(0, 66 * 10, 10))) == 1  # at most 64 shards
    assert comb([0, 10, 30], lse=0) == 1       # step 3 needs the lse
    assert comb([0, 10, 30], wsb=10) == 4
    assert lib.ce_vp_partials(ctypes.c_void_p(0x1000), 1, 1, 4, 16, _lib.i64_array((64, 16, 1)),
                              ctypes.c_void_p(0x2000), _lib.i64_array((4, 1)), 0, -100,
                              ctypes.c_void_p(0x3008), None) == 1  # partials not 16-byte aligned
    assert lib.ce_vp_partials(ctypes.c_void_p(0x1001), 1, 1, 4, 16, _lib.i64_array((64, 16, 1)),
                              ctypes.c_void_p(0x2000), _lib.i64_array((4, 1)), 0, -100,
                              ctypes.c_void_p(0x3000), None) == 1  # shard off the element size
    # the shard must lie inside the vocabulary
    assert lib.ce_vp_bwd(ctypes.c_void_p(0x1000), 1, 1, 4, 16, _lib.i64_array((64, 16, 1)),
                         ctypes.c_void_p(0x2000), _lib.i64_array((4, 1)), 40, 50,
                         ctypes.c_void_p(0x3000), 0.0, -100, 0, None, None,
                         ctypes.c_void_p(0x4000), _lib.i64_array((64, 16, 1)), None) == 1
