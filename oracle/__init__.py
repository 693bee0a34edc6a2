"""CPU oracle for the fused vocabulary cross-entropy pass (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The GPU library in ``vocabulary_cross_entropy_pass_gb300`` never
imports this package, and this package never imports that one.

The arithmetic lives in ``ce_oracle.c`` (plain C, double precision, one
OpenMP loop over rows); this module only builds it with gcc and marshals numpy
arrays through ctypes.  What each C function computes, and which web page and
section it follows, is written in that file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ce_oracle.c")
LIB = os.path.join(HERE, "libceoracle.so")

F32, BF16, F16 = 0, 1, 2
ERR_TARGET_RANGE = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    c_i64, c_dbl, c_int, c_vp = ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_void_p
    lib.oracle_ce.restype = c_int
    lib.oracle_ce.argtypes = [c_vp, c_int, c_i64, c_i64, c_i64, c_i64, c_i64, c_vp, c_i64, c_i64,
                              c_dbl, c_i64, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]
    lib.oracle_linear_ce.restype = c_int
    lib.oracle_linear_ce.argtypes = [c_vp, c_vp, c_int, c_i64, c_i64, c_i64, c_vp, c_dbl, c_i64,
                                     c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]
    lib.oracle_round.restype = c_dbl
    lib.oracle_round.argtypes = [c_dbl, c_int]
    lib.oracle_round_array.restype = None
    lib.oracle_round_array.argtypes = [c_vp, c_i64, c_int, c_vp]
    lib.oracle_encode.restype = ctypes.c_uint32
    lib.oracle_encode.argtypes = [c_dbl, c_int]
    lib.oracle_decode.restype = c_dbl
    lib.oracle_decode.argtypes = [c_vp, c_int, c_i64]
    lib.oracle_chunk_partials.restype = None
    lib.oracle_chunk_partials.argtypes = [c_vp, c_i64, c_i64, c_i64, c_vp]
    lib.oracle_combine.restype = None
    lib.oracle_combine.argtypes = [c_vp, c_int, c_vp]
    lib.oracle_num_threads.restype = c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def ce(logits: np.ndarray, dtype: int, dim0: int, dim1: int, V: int, strides=None,
       targets: np.ndarray | None = None, target_strides=None, label_smoothing: float = 0.0,
       ignore_idx: int = -100, reduce_loss: bool = False, dloss: np.ndarray | None = None,
       want_grad: bool = True, class_weights: np.ndarray | None = None, lib=None) -> dict:
    """Run the oracle on raw logits storage.

    ``logits`` is the flat storage (float32 for F32; uint16 bit patterns for BF16
    and F16), element (i, j, v) at ``i*strides[0] + j*strides[1] + v``.  Returns
    a dict with ``loss`` (N values, or one for ``reduce_loss``), ``lse`` (N),
    ``grad`` (N x V exact gradient, flattened row order; None without
    ``want_grad``), ``n`` and ``err``.
    """
    lib = lib or load()
    N = dim0 * dim1
    if strides is None:
        strides = (dim1 * V, V)
    if target_strides is None:
        target_strides = (dim1, 1)
    logits = np.ascontiguousarray(logits)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    if dloss is not None:
        dloss = np.ascontiguousarray(dloss, dtype=np.float64)
    if class_weights is not None:
        class_weights = np.ascontiguousarray(class_weights, dtype=np.float64)
        assert class_weights.shape == (V,)
    loss = np.zeros(1 if reduce_loss else N, dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    grad = np.zeros((N, V), dtype=np.float64) if want_grad else None
    n = np.zeros(1, dtype=np.int64)
    err = np.zeros(1, dtype=np.uint32)
    rc = lib.oracle_ce(_ptr(logits), dtype, dim0, dim1, V, strides[0], strides[1], _ptr(targets),
                       target_strides[0], target_strides[1], float(label_smoothing), int(ignore_idx),
                       int(bool(reduce_loss)), _ptr(dloss), _ptr(class_weights), _ptr(loss),
                       _ptr(lse), _ptr(grad), _ptr(n), _ptr(err))
    if rc != 0:
        raise MemoryError("oracle_ce ran out of host memory")
    return {"loss": loss, "lse": lse, "grad": grad, "n": int(n[0]), "err": int(err[0])}


def linear_ce(hidden: np.ndarray, weight: np.ndarray, dtype: int, N: int, H: int, V: int,
              targets: np.ndarray, label_smoothing: float = 0.0, ignore_idx: int = -100,
              reduce_loss: bool = False, dloss: np.ndarray | None = None, want_grad: bool = True,
              lib=None) -> dict:
    """lm_head + cross-entropy (see oracle_linear_ce): ``hidden`` (N*H) and
    ``weight`` (V*H) are flat storage (float32, or uint16 bits of bf16/fp16)."""
    lib = lib or load()
    hidden = np.ascontiguousarray(hidden)
    weight = np.ascontiguousarray(weight)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    if dloss is not None:
        dloss = np.ascontiguousarray(dloss, dtype=np.float64)
    loss = np.zeros(1 if reduce_loss else N, dtype=np.float64)
    gh = np.zeros((N, H), dtype=np.float64) if want_grad else None
    gw = np.zeros((V, H), dtype=np.float64) if want_grad else None
    dl = np.zeros((N, V), dtype=np.float64) if want_grad else None
    n = np.zeros(1, dtype=np.int64)
    err = np.zeros(1, dtype=np.uint32)
    rc = lib.oracle_linear_ce(_ptr(hidden), _ptr(weight), dtype, N, H, V, _ptr(targets),
                              float(label_smoothing), int(ignore_idx), int(bool(reduce_loss)),
                              _ptr(dloss), _ptr(loss), _ptr(gh), _ptr(gw), _ptr(dl), _ptr(n),
                              _ptr(err))
    if rc != 0:
        raise MemoryError("oracle_linear_ce ran out of host memory")
    return {"loss": loss, "grad_hidden": gh, "grad_weight": gw, "dlogits": dl, "n": int(n[0]),
            "err": int(err[0])}


def round_to(values, dtype: int, lib=None) -> np.ndarray:
    """Round each double to the storage format (ties to even); result as double,
    same shape as ``values``."""
    lib = lib or load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty_like(v)
    lib.oracle_round_array(_ptr(v), v.size, dtype, _ptr(out))
    return out


def encode(values, dtype: int, lib=None) -> np.ndarray:
    """Storage bits of round_to(values) (uint32 for F32, uint16 otherwise)."""
    lib = lib or load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.array([lib.oracle_encode(float(x), dtype) for x in v], dtype=np.uint64)
    return out.astype(np.uint32 if dtype == F32 else np.uint16)


def decode(storage: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Exact double value of each stored element."""
    lib = lib or load()
    s = np.ascontiguousarray(storage)
    return np.array([lib.oracle_decode(_ptr(s), dtype, k) for k in range(s.size)], dtype=np.float64)


def chunk_partials(x: np.ndarray, k0: int, k1: int, y: int, lib=None) -> np.ndarray:
    """{m, d, S, x_y, has_y} of row x (double) over columns [k0, k1)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(5, dtype=np.float64)
    lib.oracle_chunk_partials(_ptr(x), k0, k1, y, _ptr(out))
    return out


def combine(parts: np.ndarray, lib=None) -> np.ndarray:
    """{lse, x_y, S} from K chunk partials (K x 5)."""
    lib = lib or load()
    p = np.ascontiguousarray(parts, dtype=np.float64)
    out = np.zeros(3, dtype=np.float64)
    lib.oracle_combine(_ptr(p), p.shape[0], _ptr(out))
    return out


def num_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_num_threads())
