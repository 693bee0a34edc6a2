"""Fused vocabulary cross-entropy forward+backward for NVIDIA GB300 (sm_103a).

The work runs in libgbce.so (hand-written CUDA kernels behind a C ABI,
include/ce.h); this package only marshals torch tensors into that ABI.  The
entry points keep the C names:

  ce_fwd_bwd(logits, targets, ...)   loss; the gradient overwrites logits
  ce_fwd_only(logits, targets, ...)  loss (and optionally lse); logits kept
  ce_bwd(logits, targets, lse, ...)  gradient from a saved lse
  ce_workspace_bytes(...), ce_get_error(...), ce_status_string(...),
  ce_plan_path(...), ce_fwd_bwd_noalloc(...), ce_noalloc_get_error(...)

whose arguments follow the TENPU "Parallel Cross Entropy (Triton)" interface
(Ascend/TransformerEngineNPU issue #29, section 1), and
``parallel_cross_entropy`` wraps ce_fwd_only + ce_bwd in a
torch.autograd.Function with that interface's argument list.

Importing the package does not load the library; the first call does, and
raises if it is missing.  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (CE_PATH_AUTO, CE_PATH_CLUSTER, CE_PATH_ROW, CE_PATH_STREAM,
                   CE_PATH_TWO_STAGE, CE_PATH_VECROW, CE_PATH_WARP, CEError, ce_options,
                   make_options)

__all__ = ["ce_fwd_bwd", "ce_fwd_bwd_noalloc", "ce_fwd_only", "ce_bwd", "parallel_cross_entropy",
           "ce_vp_partials", "ce_vp_combine", "ce_vp_bwd", "vocab_parallel_cross_entropy",
           "ce_linear_fwd_bwd", "ce_workspace_bytes", "ce_get_error", "ce_noalloc_get_error",
           "ce_status_string",
           "ce_wait_timeout_probe",
           "ce_plan_path", "CEError", "make_options", "ce_options",
           "CE_PATH_AUTO", "CE_PATH_ROW", "CE_PATH_CLUSTER", "CE_PATH_TWO_STAGE", "CE_PATH_STREAM",
           "CE_PATH_WARP", "CE_PATH_VECROW"]

_DTYPE = {torch.float32: _lib.CE_F32, torch.bfloat16: _lib.CE_BF16, torch.float16: _lib.CE_F16}
_LAYOUT = {"bsv": _lib.CE_LAYOUT_BSV, "sbv": _lib.CE_LAYOUT_SBV}


def _dims(logits: torch.Tensor):
    if logits.dim() == 3:
        d0, d1, V = logits.shape
        s = logits.stride()
        return d0, d1, V, (s[0], s[1], s[2])
    if logits.dim() == 2:
        N, V = logits.shape
        s = logits.stride()
        return 1, N, V, (N * s[0], s[0], s[1])
    raise ValueError("logits must be (dim0, dim1, V) or (N, V)")


def _tstrides(targets: torch.Tensor, d0: int, d1: int):
    if targets.dim() == 2:
        if tuple(targets.shape) != (d0, d1):
            raise ValueError(f"targets shape {tuple(targets.shape)} does not match ({d0}, {d1})")
        return targets.stride()[0], targets.stride()[1]
    if targets.dim() == 1 and targets.shape[0] == d0 * d1 and d0 == 1:
        return d1 * targets.stride()[0], targets.stride()[0]
    raise ValueError("targets must be (dim0, dim1) (or (N,) with (N, V) logits)")


def _check(logits, targets):
    if not logits.is_cuda or not targets.is_cuda:
        raise ValueError("logits and targets must be CUDA tensors (there is no CPU path)")
    if logits.device != targets.device:
        raise ValueError("logits and targets must be on the same device")
    if logits.dtype not in _DTYPE:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if targets.dtype != torch.int64:
        raise TypeError("targets must be int64")
    if logits.stride(-1) != 1:
        raise ValueError("the vocabulary dimension must be contiguous (call .contiguous())")


def _options(opts, force_path, num_vocab_chunks, class_weights=None):
    if opts is None:
        opts = make_options(force_path=force_path, num_vocab_chunks=num_vocab_chunks)
    if class_weights is not None:
        if class_weights.dtype != torch.float32 or not class_weights.is_cuda or \
                class_weights.dim() != 1 or not class_weights.is_contiguous():
            raise TypeError("class_weights must be a contiguous float32 CUDA vector of length V")
        opts.class_weights = class_weights.data_ptr()
    return opts


def _raise(st: int, what: str):
    if st != 0:
        raise CEError(st, what)


def ce_workspace_bytes(dim0: int, dim1: int, V: int, dtype: torch.dtype, opts=None) -> int:
    lib = _lib.load()
    return int(lib.ce_workspace_bytes(dim0, dim1, V, _DTYPE[dtype],
                                      ctypes.byref(opts) if opts is not None else None))


def ce_plan_path(logits: torch.Tensor, opts=None):
    """(path, chunks) the planner picks for these logits."""
    lib = _lib.load()
    d0, d1, V, st = _dims(logits)
    chunks = ctypes.c_int(0)
    path = lib.ce_plan_path(ctypes.c_void_p(logits.data_ptr()), _DTYPE[logits.dtype], d0, d1, V,
                            _lib.i64_array(st), ctypes.byref(opts) if opts is not None else None,
                            ctypes.byref(chunks))
    return int(path), int(chunks.value)


def _workspace(workspace, d0, d1, V, dtype, opts, device):
    need = ce_workspace_bytes(d0, d1, V, dtype, opts)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def ce_fwd_bwd(logits: torch.Tensor, targets: torch.Tensor, label_smoothing: float = 0.0,
               ignore_idx: int = -100, reduce_loss: bool = False, dloss: torch.Tensor | None = None,
               layout: str = "bsv", loss_out: torch.Tensor | None = None,
               n_non_ignore_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               force_path: int = CE_PATH_AUTO, num_vocab_chunks: int = 0, opts=None,
               stream=None, class_weights: torch.Tensor | None = None) -> torch.Tensor:
    """Loss of every row (or the mean); the gradient overwrites ``logits``.

    ``dloss``: float32 CUDA tensor, one value (reduce_loss) or one per row;
    None means 1.  ``class_weights``: optional float32 CUDA vector of length V
    (torch F.cross_entropy(weight=...) semantics).  Returns ``loss_out``
    (allocated when None).
    """
    _check(logits, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(logits)
    ts = _tstrides(targets, d0, d1)
    opts = _options(opts, force_path, num_vocab_chunks, class_weights)
    dev = logits.device
    if loss_out is None:
        loss_out = torch.empty(1 if reduce_loss else d0 * d1, dtype=torch.float32, device=dev)
    if dloss is not None and (dloss.dtype != torch.float32 or not dloss.is_cuda):
        raise TypeError("dloss must be a float32 CUDA tensor")
    ws, wsb = _workspace(workspace, d0, d1, V, logits.dtype, opts, dev)
    rc = lib.ce_fwd_bwd(ctypes.c_void_p(logits.data_ptr()), _DTYPE[logits.dtype], _LAYOUT[layout],
                        d0, d1, V, _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()),
                        _lib.i64_array(ts), float(label_smoothing), int(ignore_idx),
                        int(bool(reduce_loss)),
                        ctypes.c_void_p(dloss.data_ptr() if dloss is not None else None),
                        ctypes.c_void_p(loss_out.data_ptr()), ctypes.c_void_p(logits.data_ptr()),
                        ctypes.c_void_p(n_non_ignore_out.data_ptr()
                                        if n_non_ignore_out is not None else None),
                        ctypes.c_void_p(ws.data_ptr()), wsb, ctypes.byref(opts),
                        _stream(dev, stream))
    _raise(rc, "ce_fwd_bwd")
    return loss_out


def ce_fwd_only(logits: torch.Tensor, targets: torch.Tensor, label_smoothing: float = 0.0,
                ignore_idx: int = -100, reduce_loss: bool = False, layout: str = "bsv",
                loss_out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
                n_non_ignore_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                force_path: int = CE_PATH_AUTO, num_vocab_chunks: int = 0, opts=None,
                stream=None, class_weights: torch.Tensor | None = None) -> torch.Tensor:
    """Loss of every row (or the mean); ``logits`` is left untouched."""
    _check(logits, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(logits)
    ts = _tstrides(targets, d0, d1)
    opts = _options(opts, force_path, num_vocab_chunks, class_weights)
    dev = logits.device
    if loss_out is None:
        loss_out = torch.empty(1 if reduce_loss else d0 * d1, dtype=torch.float32, device=dev)
    ws, wsb = _workspace(workspace, d0, d1, V, logits.dtype, opts, dev)
    rc = lib.ce_fwd_only(ctypes.c_void_p(logits.data_ptr()), _DTYPE[logits.dtype], _LAYOUT[layout],
                         d0, d1, V, _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()),
                         _lib.i64_array(ts), float(label_smoothing), int(ignore_idx),
                         int(bool(reduce_loss)), ctypes.c_void_p(loss_out.data_ptr()),
                         ctypes.c_void_p(lse_out.data_ptr() if lse_out is not None else None),
                         ctypes.c_void_p(n_non_ignore_out.data_ptr()
                                         if n_non_ignore_out is not None else None),
                         ctypes.c_void_p(ws.data_ptr()), wsb, ctypes.byref(opts),
                         _stream(dev, stream))
    _raise(rc, "ce_fwd_only")
    return loss_out


def ce_fwd_bwd_noalloc(logits: torch.Tensor, targets: torch.Tensor, loss_out: torch.Tensor,
                       label_smoothing: float = 0.0, ignore_idx: int = -100,
                       reduce_loss: bool = False, dloss: torch.Tensor | None = None,
                       layout: str = "bsv", n_non_ignore_out: torch.Tensor | None = None,
                       opts=None, stream=None) -> torch.Tensor:
    """ce_fwd_bwd for callers that cannot hand out device memory: the pass
    keeps its scratch in the library's own fixed device array, so nothing is
    allocated here either (``loss_out`` must be given).  Calls that may
    overlap on the GPU share that array and must be serialised."""
    _check(logits, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(logits)
    ts = _tstrides(targets, d0, d1)
    opts = _options(opts, CE_PATH_AUTO, 0)
    rc = lib.ce_fwd_bwd_noalloc(
        ctypes.c_void_p(logits.data_ptr()), _DTYPE[logits.dtype], _LAYOUT[layout], d0, d1, V,
        _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()), _lib.i64_array(ts),
        float(label_smoothing), int(ignore_idx), int(bool(reduce_loss)),
        ctypes.c_void_p(dloss.data_ptr() if dloss is not None else None),
        ctypes.c_void_p(loss_out.data_ptr()), ctypes.c_void_p(logits.data_ptr()),
        ctypes.c_void_p(n_non_ignore_out.data_ptr() if n_non_ignore_out is not None else None),
        ctypes.byref(opts), _stream(logits.device, stream))
    if rc == 4:
        raise CEError(rc, "ce_fwd_bwd_noalloc: the problem needs more scratch than the "
                          "library's fixed 2 MiB array holds")
    _raise(rc, "ce_fwd_bwd_noalloc")
    return loss_out


def ce_get_error(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    """(status, device error word) of the last pass that used ``workspace``;
    waits for the stream."""
    lib = _lib.load()
    err = ctypes.c_uint32(0)
    rc = lib.ce_get_error(ctypes.c_void_p(workspace.data_ptr()), _stream(workspace.device, stream),
                          ctypes.byref(err))
    return int(rc), int(err.value)


def ce_noalloc_get_error(device=None, stream=None) -> tuple[int, int]:
    """(status, device error word) of the last ce_fwd_bwd_noalloc pass on
    ``device`` (default: the current CUDA device); waits for the stream."""
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    err = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        rc = lib.ce_noalloc_get_error(_stream(dev, stream), ctypes.byref(err))
    return int(rc), int(err.value)


def ce_wait_timeout_probe(workspace: torch.Tensor, stream=None) -> None:
    """Run the kernels' bounded wait once on a barrier nothing completes; its
    timeout lands in ``workspace``'s error word (read it with ce_get_error,
    ~1.5 s later)."""
    if not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    lib = _lib.load()
    nbytes = workspace.numel() * workspace.element_size()
    _raise(lib.ce_wait_timeout_probe(ctypes.c_void_p(workspace.data_ptr()), nbytes,
                                     _stream(workspace.device, stream)), "ce_wait_timeout_probe")


def ce_status_string(status: int) -> str:
    return _lib.load().ce_status_string(int(status)).decode()



def ce_bwd(logits: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
           label_smoothing: float = 0.0, ignore_idx: int = -100, reduce_loss: bool = False,
           dloss: torch.Tensor | None = None, n_non_ignore: torch.Tensor | None = None,
           grad: torch.Tensor | None = None, layout: str = "bsv", stream=None) -> torch.Tensor:
    """Gradient of the cross-entropy from the ``lse`` a forward-only pass saved.
    ``grad`` may be ``logits`` itself (in place) or a separate tensor of the
    same shape and dtype (allocated when None).  ``n_non_ignore`` (int64 CUDA
    tensor from the forward) is needed for reduce_loss."""
    _check(logits, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(logits)
    ts = _tstrides(targets, d0, d1)
    if grad is None:
        grad = torch.empty_like(logits)
    if grad.shape != logits.shape or grad.dtype != logits.dtype or not grad.is_cuda:
        raise ValueError("grad must match logits in shape and dtype, on the GPU")
    gst = _dims(grad)[3]
    for tens, name in ((lse, "lse"), (dloss, "dloss")):
        if tens is not None and (tens.dtype != torch.float32 or not tens.is_cuda):
            raise TypeError(f"{name} must be a float32 CUDA tensor")
    rc = lib.ce_bwd(ctypes.c_void_p(logits.data_ptr()), _DTYPE[logits.dtype], _LAYOUT[layout], d0,
                    d1, V, _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()),
                    _lib.i64_array(ts), ctypes.c_void_p(lse.data_ptr()), float(label_smoothing),
                    int(ignore_idx), int(bool(reduce_loss)),
                    ctypes.c_void_p(dloss.data_ptr() if dloss is not None else None),
                    ctypes.c_void_p(n_non_ignore.data_ptr() if n_non_ignore is not None else None),
                    ctypes.c_void_p(grad.data_ptr()), _lib.i64_array(gst),
                    _stream(logits.device, stream))
    _raise(rc, "ce_bwd")
    return grad


class _ParallelCrossEntropy(torch.autograd.Function):
    """Forward: ce_fwd_only (loss, lse and the kept-row count saved).
    Backward: ce_bwd with the upstream gradient, into a new tensor or, with
    ``inplace_grad``, over the logits (the in-place staging of TENPU #29
    section 6: the caller gives up the logits)."""

    @staticmethod
    def forward(ctx, inp, target, label_smoothing, reduce_loss, ignore_idx, layout, inplace_grad):
        x = inp if inp.stride(-1) == 1 else inp.contiguous()
        d0, d1, V, _ = _dims(x)
        lse = torch.empty(d0 * d1, dtype=torch.float32, device=x.device)
        n = torch.empty(1, dtype=torch.int64, device=x.device)
        loss = ce_fwd_only(x, target, label_smoothing=label_smoothing, ignore_idx=ignore_idx,
                           reduce_loss=reduce_loss, layout=layout, lse_out=lse,
                           n_non_ignore_out=n)
        ctx.save_for_backward(x, target, lse, n)
        ctx.cfg = (label_smoothing, reduce_loss, ignore_idx, layout, inplace_grad)
        return loss.view(()) if reduce_loss else loss.view(target.shape)

    @staticmethod
    def backward(ctx, grad_out):
        x, target, lse, n = ctx.saved_tensors
        a, reduce_loss, ignore_idx, layout, inplace_grad = ctx.cfg
        dl = grad_out.detach().to(torch.float32).contiguous().reshape(-1)
        g = ce_bwd(x, target, lse, label_smoothing=a, ignore_idx=ignore_idx,
                   reduce_loss=reduce_loss, dloss=dl, n_non_ignore=n,
                   grad=x if inplace_grad else None, layout=layout)
        return g, None, None, None, None, None, None


def parallel_cross_entropy(inp: torch.Tensor, target: torch.Tensor, label_smoothing: float = 0.0,
                           reduce_loss: bool = False, dist_process_group=None,
                           ignore_idx: int = -100, layout: str = "bsv",
                           inplace_grad: bool = False) -> torch.Tensor:
    """Cross-entropy with autograd, argument list of TENPU #29 section 1.
    Returns the per-token loss (shape of ``target``) or the mean over kept
    tokens (``reduce_loss``); ``backward`` fills ``inp.grad`` through ce_bwd.
    One GPU only: ``dist_process_group`` must be None."""
    if dist_process_group is not None:
        raise NotImplementedError("vocabulary-parallel process groups are not supported: one GPU")
    return _ParallelCrossEntropy.apply(inp, target, label_smoothing, reduce_loss, ignore_idx,
                                       layout, inplace_grad)


# ---------------------------------------------------------------- vocabulary parallel
def ce_vp_partials(shard: torch.Tensor, targets: torch.Tensor, vocab_offset: int,
                   partials: torch.Tensor | None = None, ignore_idx: int = -100,
                   stream=None) -> torch.Tensor:
    """Step 1: (max, sum-exp, sum, target logit) per row of one vocabulary
    shard; returns a float32 (N, 4) tensor."""
    _check(shard, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(shard)
    ts = _tstrides(targets, d0, d1)
    if partials is None:
        partials = torch.empty(d0 * d1, 4, dtype=torch.float32, device=shard.device)
    rc = lib.ce_vp_partials(ctypes.c_void_p(shard.data_ptr()), _DTYPE[shard.dtype], d0, d1, V,
                            _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()),
                            _lib.i64_array(ts), int(vocab_offset), int(ignore_idx),
                            ctypes.c_void_p(partials.data_ptr()), _stream(shard.device, stream))
    _raise(rc, "ce_vp_partials")
    return partials


def ce_vp_combine(partials: torch.Tensor, shard_offsets, targets: torch.Tensor,
                  label_smoothing: float = 0.0, ignore_idx: int = -100, reduce_loss: bool = False,
                  loss_out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
                  n_non_ignore_out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None):
    """Step 2: combine (R, N, 4) partials in shard order; returns (loss, lse)."""
    lib = _lib.load()
    R = partials.shape[0]
    if targets.dim() != 2:
        raise ValueError("targets must be (dim0, dim1)")
    d0, d1 = targets.shape
    ts = targets.stride()
    dev = targets.device
    V = int(shard_offsets[-1])
    if loss_out is None:
        loss_out = torch.empty(1 if reduce_loss else d0 * d1, dtype=torch.float32, device=dev)
    if lse_out is None:
        lse_out = torch.empty(d0 * d1, dtype=torch.float32, device=dev)
    ws, wsb = _workspace(workspace, d0, d1, V, torch.float32, None, dev)
    rc = lib.ce_vp_combine(ctypes.c_void_p(partials.contiguous().data_ptr()), R,
                           _lib.i64_array(shard_offsets), d0, d1,
                           ctypes.c_void_p(targets.data_ptr()), _lib.i64_array(ts),
                           float(label_smoothing), int(ignore_idx), int(bool(reduce_loss)),
                           ctypes.c_void_p(loss_out.data_ptr()), ctypes.c_void_p(lse_out.data_ptr()),
                           ctypes.c_void_p(n_non_ignore_out.data_ptr()
                                           if n_non_ignore_out is not None else None),
                           ctypes.c_void_p(ws.data_ptr()), wsb, _stream(dev, stream))
    _raise(rc, "ce_vp_combine")
    return loss_out, lse_out


def ce_vp_bwd(shard: torch.Tensor, targets: torch.Tensor, vocab_offset: int, V_total: int,
              lse: torch.Tensor, label_smoothing: float = 0.0, ignore_idx: int = -100,
              reduce_loss: bool = False, dloss: torch.Tensor | None = None,
              n_non_ignore: torch.Tensor | None = None, grad: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Step 3: the gradient of one shard (in place when ``grad`` is ``shard``)."""
    _check(shard, targets)
    lib = _lib.load()
    d0, d1, V, st = _dims(shard)
    ts = _tstrides(targets, d0, d1)
    if grad is None:
        grad = torch.empty_like(shard)
    gst = _dims(grad)[3]
    rc = lib.ce_vp_bwd(ctypes.c_void_p(shard.data_ptr()), _DTYPE[shard.dtype], d0, d1, V,
                       _lib.i64_array(st), ctypes.c_void_p(targets.data_ptr()), _lib.i64_array(ts),
                       int(vocab_offset), int(V_total), ctypes.c_void_p(lse.data_ptr()),
                       float(label_smoothing), int(ignore_idx), int(bool(reduce_loss)),
                       ctypes.c_void_p(dloss.data_ptr() if dloss is not None else None),
                       ctypes.c_void_p(n_non_ignore.data_ptr() if n_non_ignore is not None else None),
                       ctypes.c_void_p(grad.data_ptr()), _lib.i64_array(gst),
                       _stream(shard.device, stream))
    _raise(rc, "ce_vp_bwd")
    return grad


def vocab_parallel_cross_entropy(shards, targets: torch.Tensor, label_smoothing: float = 0.0,
                                 ignore_idx: int = -100, reduce_loss: bool = False,
                                 dloss: torch.Tensor | None = None, inplace_grad: bool = True):
    """All three steps over vocabulary shards held by one GPU (shard k holds
    the next block of columns).  Returns (loss, gradients per shard); with
    ``inplace_grad`` the gradients overwrite the shards."""
    offsets = [0]
    for sh in shards:
        offsets.append(offsets[-1] + sh.shape[-1])
    N = targets.numel()
    dev = targets.device
    part = torch.empty(len(shards), N, 4, dtype=torch.float32, device=dev)
    for k, sh in enumerate(shards):
        ce_vp_partials(sh, targets, offsets[k], partials=part[k], ignore_idx=ignore_idx)
    n = torch.empty(1, dtype=torch.int64, device=dev)
    loss, lse = ce_vp_combine(part, offsets, targets, label_smoothing=label_smoothing,
                              ignore_idx=ignore_idx, reduce_loss=reduce_loss, n_non_ignore_out=n)
    grads = [ce_vp_bwd(sh, targets, offsets[k], offsets[-1], lse, label_smoothing=label_smoothing,
                       ignore_idx=ignore_idx, reduce_loss=reduce_loss, dloss=dloss,
                       n_non_ignore=n, grad=sh if inplace_grad else None)
             for k, sh in enumerate(shards)]
    return loss, grads


# ---------------------------------------------------------------- lm_head + cross-entropy
def ce_linear_fwd_bwd(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                      label_smoothing: float = 0.0, ignore_idx: int = -100,
                      reduce_loss: bool = False, dloss: torch.Tensor | None = None,
                      grad_hidden: torch.Tensor | bool | None = True,
                      grad_weight: torch.Tensor | bool | None = True, chunk_rows: int = 4096,
                      loss_out: torch.Tensor | None = None,
                      n_non_ignore_out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """lm_head (hidden (N, H) . weight (V, H)^T) + cross-entropy, chunk_rows
    rows at a time: the (N, V) logits never exist.  ``grad_hidden``: a (N, H)
    tensor of the input dtype to write, True to allocate one, None to skip;
    ``grad_weight``: a float32 (V, H) tensor accumulated into, True to
    allocate a zeroed one, None to skip.  Returns (loss, grad_hidden,
    grad_weight)."""
    if not (hidden.is_cuda and weight.is_cuda and targets.is_cuda):
        raise ValueError("hidden, weight and targets must be CUDA tensors (there is no CPU path)")
    if hidden.dtype not in _DTYPE or weight.dtype != hidden.dtype:
        raise TypeError("hidden and weight must share a float32/bfloat16/float16 dtype")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden (N, H) and weight (V, H) expected")
    hidden = hidden.contiguous()
    weight = weight.contiguous()
    t = targets.reshape(-1).contiguous()
    if t.dtype != torch.int64 or t.numel() != hidden.shape[0]:
        raise ValueError("targets must be int64 with one entry per hidden row")
    lib = _lib.load()
    N, H = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    if grad_hidden is True:
        grad_hidden = torch.empty_like(hidden)
    if grad_weight is True:
        grad_weight = torch.zeros(V, H, dtype=torch.float32, device=dev)
    if grad_weight is not None and grad_weight is not False and grad_weight.dtype != torch.float32:
        raise TypeError("grad_weight accumulates in float32")
    gh = grad_hidden if isinstance(grad_hidden, torch.Tensor) else None
    gw = grad_weight if isinstance(grad_weight, torch.Tensor) else None
    if loss_out is None:
        loss_out = torch.empty(1 if reduce_loss else N, dtype=torch.float32, device=dev)
    need = int(lib.ce_linear_workspace_bytes(N, H, V, _DTYPE[hidden.dtype], int(chunk_rows)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rc = lib.ce_linear_fwd_bwd(
        ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(weight.data_ptr()),
        _DTYPE[hidden.dtype], N, H, V, ctypes.c_void_p(t.data_ptr()), float(label_smoothing),
        int(ignore_idx), int(bool(reduce_loss)),
        ctypes.c_void_p(dloss.data_ptr() if dloss is not None else None),
        ctypes.c_void_p(loss_out.data_ptr()),
        ctypes.c_void_p(gh.data_ptr() if gh is not None else None),
        ctypes.c_void_p(gw.data_ptr() if gw is not None else None),
        ctypes.c_void_p(n_non_ignore_out.data_ptr() if n_non_ignore_out is not None else None),
        int(chunk_rows), ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel() * workspace.element_size(), _stream(dev, stream))
    _raise(rc, "ce_linear_fwd_bwd")
    return loss_out, gh, gw
