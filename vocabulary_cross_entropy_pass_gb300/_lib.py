"""ctypes binding of libgbce (include/ce.h).

Argument marshalling only: tensors become device pointers, shapes and
strides; every step of the pass runs in the library's CUDA kernels.  There is
no CPU path: a tensor that is not on a CUDA device, or a library that was not
built, raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgbce.so")

CE_F32, CE_BF16, CE_F16 = 0, 1, 2
CE_LAYOUT_BSV, CE_LAYOUT_SBV = 0, 1
(CE_PATH_AUTO, CE_PATH_ROW, CE_PATH_CLUSTER, CE_PATH_TWO_STAGE, CE_PATH_STREAM, CE_PATH_WARP,
 CE_PATH_VECROW) = (0, 1, 2, 3, 4, 5, 6)
CE_DEVERR_TARGET_RANGE, CE_DEVERR_TIMEOUT = 0x1, 0x2

STATUS = {
    0: "CE_OK",
    1: "CE_ERR_INVALID_ARG",
    2: "CE_ERR_UNSUPPORTED_DTYPE",
    3: "CE_ERR_BAD_STRIDE",
    4: "CE_ERR_WORKSPACE_TOO_SMALL",
    5: "CE_ERR_LAUNCH",
    6: "CE_ERR_TARGET_RANGE",
    7: "CE_ERR_DEVICE_TIMEOUT",
    8: "CE_ERR_UNSUPPORTED_PATH",
}

# every function include/ce.h declares
EXPORTS = ("ce_workspace_bytes", "ce_fwd_bwd", "ce_fwd_only", "ce_get_error", "ce_status_string",
           "ce_plan_path", "ce_fwd_bwd_noalloc", "ce_bwd", "ce_vp_partials", "ce_vp_combine",
           "ce_vp_bwd", "ce_linear_workspace_bytes", "ce_linear_fwd_bwd", "ce_wait_timeout_probe",
           "ce_noalloc_get_error")


class ce_options(ctypes.Structure):
    _fields_ = [
        ("force_path", ctypes.c_int),
        ("num_vocab_chunks", ctypes.c_int),
        ("event_begin", ctypes.c_void_p),
        ("event_end", ctypes.c_void_p),
        ("tune_threads", ctypes.c_int),
        ("tune_stages", ctypes.c_int),
        ("tune_ctas_per_sm", ctypes.c_int),
        ("tune_l2_keep", ctypes.c_int),
        ("tune_tile_kb", ctypes.c_int),
        ("class_weights", ctypes.c_void_p),
        ("reserved", ctypes.c_int * 2),
    ]


class CEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {name}" if what else name)


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libgbce.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        I64_3 = ctypes.POINTER(ctypes.c_int64)
        opt_p = ctypes.POINTER(ce_options)
        lib.ce_workspace_bytes.restype = ctypes.c_size_t
        lib.ce_workspace_bytes.argtypes = [i64, i64, i64, i32, opt_p]
        lib.ce_fwd_bwd.restype = i32
        lib.ce_fwd_bwd.argtypes = [vp, i32, i32, i64, i64, i64, I64_3, vp, I64_3, f32, i64, i32, vp,
                                   vp, vp, vp, vp, ctypes.c_size_t, opt_p, vp]
        lib.ce_fwd_only.restype = i32
        lib.ce_fwd_only.argtypes = [vp, i32, i32, i64, i64, i64, I64_3, vp, I64_3, f32, i64, i32,
                                    vp, vp, vp, vp, ctypes.c_size_t, opt_p, vp]
        lib.ce_fwd_bwd_noalloc.restype = i32
        lib.ce_fwd_bwd_noalloc.argtypes = [vp, i32, i32, i64, i64, i64, I64_3, vp, I64_3, f32, i64,
                                           i32, vp, vp, vp, vp, opt_p, vp]
        lib.ce_bwd.restype = i32
        lib.ce_bwd.argtypes = [vp, i32, i32, i64, i64, i64, I64_3, vp, I64_3, vp, f32, i64, i32, vp,
                               vp, vp, I64_3, vp]
        lib.ce_vp_partials.restype = i32
        lib.ce_vp_partials.argtypes = [vp, i32, i64, i64, i64, I64_3, vp, I64_3, i64, i64, vp, vp]
        lib.ce_vp_combine.restype = i32
        lib.ce_vp_combine.argtypes = [vp, i32, I64_3, i64, i64, vp, I64_3, f32, i64, i32, vp, vp,
                                      vp, vp, ctypes.c_size_t, vp]
        lib.ce_vp_bwd.restype = i32
        lib.ce_vp_bwd.argtypes = [vp, i32, i64, i64, i64, I64_3, vp, I64_3, i64, i64, vp, f32, i64,
                                  i32, vp, vp, vp, I64_3, vp]
        lib.ce_linear_workspace_bytes.restype = ctypes.c_size_t
        lib.ce_linear_workspace_bytes.argtypes = [i64, i64, i64, i32, i64]
        lib.ce_linear_fwd_bwd.restype = i32
        lib.ce_linear_fwd_bwd.argtypes = [vp, vp, i32, i64, i64, i64, vp, f32, i64, i32, vp, vp, vp,
                                          vp, vp, i64, vp, ctypes.c_size_t, vp]
        lib.ce_wait_timeout_probe.restype = i32
        lib.ce_wait_timeout_probe.argtypes = [vp, ctypes.c_size_t, vp]
        lib.ce_get_error.restype = i32
        lib.ce_get_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.ce_noalloc_get_error.restype = i32
        lib.ce_noalloc_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.ce_status_string.restype = ctypes.c_char_p
        lib.ce_status_string.argtypes = [i32]
        lib.ce_plan_path.restype = i32
        lib.ce_plan_path.argtypes = [vp, i32, i64, i64, i64, I64_3, opt_p, ctypes.POINTER(i32)]
        _lib = lib
        return lib


def i64_array(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def make_options(force_path: int = 0, num_vocab_chunks: int = 0, event_begin=None, event_end=None,
                 tune_threads: int = 0, tune_stages: int = 0, tune_ctas_per_sm: int = 0,
                 tune_l2_keep: int = 0, tune_tile_kb: int = 0, class_weights=None):
    o = ce_options()
    o.force_path = force_path
    o.num_vocab_chunks = num_vocab_chunks
    o.event_begin = event_begin
    o.event_end = event_end
    o.tune_threads = tune_threads
    o.tune_stages = tune_stages
    o.tune_ctas_per_sm = tune_ctas_per_sm
    o.tune_l2_keep = tune_l2_keep
    o.tune_tile_kb = tune_tile_kb
    o.class_weights = class_weights  # device address (int) or None
    return o
