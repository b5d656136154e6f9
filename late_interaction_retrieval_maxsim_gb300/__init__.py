"""GB300-native fused MaxSim (late-interaction scoring).

Python binding of ``libmaxsim.so`` (C ABI in ``include/maxsim.h``).  This
module only marshals torch tensors into the C calls -- allocating outputs
and workspaces with torch, passing data pointers and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU or PyTorch fallback: if the library is not built or no GPU
is present, the calls raise.

Entry points (same names as the C ABI):
  maxsim_forward   -- fused forward (FP16/BF16/INT8, dense or packed docs)
  maxsim_backward  -- dQ, dD from the saved argmax (inverse-grid CSR)
  maxsim_build_csr -- the inverse-grid CSR itself
  maxsim_forward_noalloc -- the forward with library-owned scratch
  maxsim_forward_host -- the forward over a host-resident corpus, streamed
                         to the device in blocks (out-of-core scoring)
  maxsim_forward_int8_per_token -- INT8 forward with one scale per token
  maxsim_topk      -- row-wise top-K selection (ties to the lower column)
  maxsim_rerank_two_stage -- INT8 scan, top-K' candidates, FP16 rescoring
  maxsim_chamfer_forward / maxsim_chamfer_backward / maxsim_chamfer_build_csr
                   -- the Chamfer distance on the same skeleton
  maxsim_forward_with_counts / maxsim_backward_with_counts
                   -- the training pair under its earlier names (now the
                      same as maxsim_forward / maxsim_backward: the backward
                      sorts each document's sources itself)
  maxsim_probe_l2_read -- a plain L2-resident read (the backward's roofline)
  maxsim_device_status, maxsim_forward_workspace_size,
  maxsim_backward_workspace_size, maxsim_abi_version
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "load_library", "library_path", "maxsim_forward", "maxsim_backward", "maxsim_build_csr",
    "maxsim_device_status", "maxsim_forward_workspace_size", "maxsim_backward_workspace_size",
    "maxsim_abi_version", "maxsim_forward_noalloc", "maxsim_forward_host",
    "maxsim_forward_host_workspace_size", "maxsim_forward_int8_per_token", "maxsim_topk",
    "maxsim_rerank_two_stage", "maxsim_rerank_workspace_size", "maxsim_chamfer_forward",
    "maxsim_chamfer_backward", "maxsim_chamfer_build_csr", "maxsim_forward_with_counts",
    "maxsim_backward_with_counts", "maxsim_selftest_bounded_wait", "maxsim_forward_plan", "maxsim_probe_l2_read",
    "MaxSimError",
    "DTYPE_CODES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None

STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace",
                4: "cuda error", 5: "device fault"}


class MaxSimError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


def library_path() -> str:
    return os.path.join(_PKG, "libmaxsim.so")


def load_library():
    """Load the in-tree ``libmaxsim.so`` (built by ``__graft_entry__.build()``
    or ``python -m late_interaction_retrieval_maxsim_gb300._build``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    lib.maxsim_abi_version.argtypes = []
    lib.maxsim_abi_version.restype = i32
    lib.maxsim_status_string.argtypes = [ctypes.c_int]
    lib.maxsim_status_string.restype = ctypes.c_char_p
    lib.maxsim_forward_workspace_size.argtypes = [i32, i32, i32, i32, ctypes.c_int]
    lib.maxsim_forward_workspace_size.restype = sz
    lib.maxsim_forward.argtypes = [vp, vp, i32, i32, vp, vp, i32, i64, i32, ctypes.c_int, f32, f32,
                                   vp, vp, vp, vp, sz, vp]
    lib.maxsim_forward.restype = ctypes.c_int
    lib.maxsim_backward_workspace_size.argtypes = [i32, i32, i32, i64]
    lib.maxsim_backward_workspace_size.restype = sz
    lib.maxsim_build_csr.argtypes = [vp, vp, i32, i32, vp, i32, i64, vp, vp, vp, sz, vp]
    lib.maxsim_build_csr.restype = ctypes.c_int
    lib.maxsim_backward.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, i32, i64, i32, ctypes.c_int,
                                    vp, vp, vp, sz, vp]
    lib.maxsim_backward.restype = ctypes.c_int
    lib.maxsim_forward_noalloc.argtypes = [vp, vp, i32, i32, vp, vp, i32, i64, i32, ctypes.c_int, f32, f32,
                                           vp, vp, vp, vp]
    lib.maxsim_forward_noalloc.restype = ctypes.c_int
    lib.maxsim_forward_host_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32, ctypes.c_int]
    lib.maxsim_forward_host_workspace_size.restype = sz
    lib.maxsim_forward_host.argtypes = [vp, vp, i32, i32, vp, vp, i32, i64, i32, ctypes.c_int, f32, f32,
                                        vp, vp, vp, i32, i64, vp, sz, vp, vp]
    lib.maxsim_forward_host.restype = ctypes.c_int
    lib.maxsim_forward_int8_per_token.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, i32, i64, i32, vp, vp,
                                                  vp, sz, vp]
    lib.maxsim_forward_int8_per_token.restype = ctypes.c_int
    lib.maxsim_topk.argtypes = [vp, i32, i32, i64, i32, vp, vp, vp]
    lib.maxsim_topk.restype = ctypes.c_int
    lib.maxsim_rerank_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_int]
    lib.maxsim_rerank_workspace_size.restype = sz
    lib.maxsim_rerank_two_stage.argtypes = [vp, vp, f32, vp, vp, f32, vp, vp, ctypes.c_int, vp, i32, i32, vp,
                                            i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.maxsim_rerank_two_stage.restype = ctypes.c_int
    lib.maxsim_chamfer_forward_workspace_size.argtypes = [i32, i64, i64, i32, i32]
    lib.maxsim_chamfer_forward_workspace_size.restype = sz
    lib.maxsim_chamfer_forward.argtypes = [vp, vp, vp, vp, i32, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.maxsim_chamfer_forward.restype = ctypes.c_int
    lib.maxsim_chamfer_csr_workspace_size.argtypes = [i64, i64]
    lib.maxsim_chamfer_csr_workspace_size.restype = sz
    lib.maxsim_chamfer_build_csr.argtypes = [vp, vp, vp, i32, i64, i64, vp, vp, vp, sz, vp]
    lib.maxsim_chamfer_build_csr.restype = ctypes.c_int
    lib.maxsim_chamfer_backward_workspace_size.argtypes = [i64, i64]
    lib.maxsim_chamfer_backward_workspace_size.restype = sz
    lib.maxsim_chamfer_backward.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, vp, vp, vp, vp, vp, sz, vp]
    lib.maxsim_chamfer_backward.restype = ctypes.c_int
    lib.maxsim_forward_with_counts.argtypes = [vp, vp, i32, i32, vp, vp, i32, i64, i32, ctypes.c_int, vp, vp,
                                               vp, sz, vp, sz, vp]
    lib.maxsim_forward_with_counts.restype = ctypes.c_int
    lib.maxsim_backward_with_counts.argtypes = lib.maxsim_backward.argtypes
    lib.maxsim_backward_with_counts.restype = ctypes.c_int
    lib.maxsim_device_status.argtypes = [vp, i32, ctypes.POINTER(i32)]
    lib.maxsim_device_status.restype = ctypes.c_int
    lib.maxsim_probe_l2_read.argtypes = [vp, sz, i32, vp, vp]
    lib.maxsim_probe_l2_read.restype = ctypes.c_int
    lib.maxsim_selftest_bounded_wait.argtypes = [ctypes.c_uint32, vp]
    lib.maxsim_selftest_bounded_wait.restype = ctypes.c_int
    lib.maxsim_forward_plan.argtypes = [i32, i32, i32, i64, ctypes.c_int, i32, i32, ctypes.POINTER(i32)]
    lib.maxsim_forward_plan.restype = ctypes.c_int
    _LIB = lib
    return lib


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    codes = {torch.float16: 0, torch.bfloat16: 1, torch.int8: 2}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


DTYPE_CODES = {"fp16": 0, "bf16": 1, "int8": 2}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        msg = load_library().maxsim_status_string(status).decode()
        raise MaxSimError(fn, status, msg)


def _require(t, name, dtype=None, device=None, contiguous=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _check_qd(Q, D):
    """Shapes of a forward's Q [n_q, lq_max, dim] and D [total, dim]."""
    torch = _torch()
    if not isinstance(Q, torch.Tensor) or not isinstance(D, torch.Tensor):
        raise TypeError("Q and D must be tensors")
    if Q.dim() != 3 or D.dim() != 2 or Q.shape[2] != D.shape[1]:
        raise ValueError("Q must be [n_q, lq_max, dim] and D [total, dim]")


def _check_output(t, name, shape, dtype, device):
    """A caller-provided output: exactly the shape, dtype and device the
    kernels write (they index it without bounds), contiguous."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _check_forward_outputs(n_q, n_docs, lq_max, device, scores, argmax, raw_scores):
    torch = _torch()
    _check_output(scores, "scores", (n_q, n_docs), torch.float32, device)
    if argmax is not None:
        _check_output(argmax, "argmax", (n_q, n_docs, lq_max), torch.int32, device)
    if raw_scores is not None:
        _check_output(raw_scores, "raw_scores", (n_q, n_docs), torch.int64, device)


def maxsim_abi_version() -> int:
    return int(load_library().maxsim_abi_version())


def maxsim_forward_workspace_size(n_q: int, lq_max: int, n_docs: int, dtype, dim: int = 128) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return int(load_library().maxsim_forward_workspace_size(n_q, lq_max, n_docs, dim, code))


def maxsim_backward_workspace_size(n_q: int, lq_max: int, n_docs: int, total_d_tokens: int) -> int:
    return int(load_library().maxsim_backward_workspace_size(n_q, lq_max, n_docs, total_d_tokens))


def maxsim_forward(Q, q_lens, D, cu_seqlens, *, with_argmax: bool = True, q_scale: float = 1.0,
                   d_scale: float = 1.0, scores=None, argmax=None, raw_scores=None, workspace=None,
                   want_raw: bool = False, stream=None):
    """Fused MaxSim forward (C: ``maxsim_forward``).

    Q [n_q, lq_max, 128] and D [total, 128] of the same dtype (float16,
    bfloat16 or int8); q_lens [n_q] and cu_seqlens [n_docs+1] int32 on the
    same device.  Returns (scores [n_q, n_docs] float32, argmax [n_q, n_docs,
    lq_max] int32 or None, raw_scores [n_q, n_docs] int64 or None)."""
    torch = _torch()
    lib = load_library()
    _check_qd(Q, D)
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    total = D.shape[0]
    # caller-provided outputs are written without bounds checks
    if scores is not None:
        _check_output(scores, "scores", (n_q, n_docs), torch.float32, Q.device)
    if argmax is not None and with_argmax:
        _check_output(argmax, "argmax", (n_q, n_docs, lq_max), torch.int32, Q.device)
    _require(Q, "Q")
    dev = Q.device
    _require(D, "D", dtype=Q.dtype, device=dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if q_lens.shape != (n_q,):
        raise ValueError(f"q_lens must have shape ({n_q},)")
    code = _dtype_code(Q)
    if scores is None:
        scores = torch.empty((n_q, n_docs), dtype=torch.float32, device=dev)
    if with_argmax and argmax is None:
        argmax = torch.empty((n_q, n_docs, lq_max), dtype=torch.int32, device=dev)
    if not with_argmax:
        argmax = None
    if code == 2 and want_raw and raw_scores is None:
        raw_scores = torch.empty((n_q, n_docs), dtype=torch.int64, device=dev)
    if code != 2:
        raw_scores = None
    _check_forward_outputs(n_q, n_docs, lq_max, dev, scores, argmax, raw_scores)
    ws_bytes = maxsim_forward_workspace_size(n_q, lq_max, n_docs, code, dim)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_forward(_ptr(Q), _ptr(q_lens), n_q, lq_max, _ptr(D), _ptr(cu_seqlens), n_docs,
                                total, dim, code, float(q_scale), float(d_scale), _ptr(scores),
                                _ptr(raw_scores), _ptr(argmax), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("maxsim_forward", st)
    return scores, argmax, raw_scores


def maxsim_forward_noalloc(Q, q_lens, D, cu_seqlens, scores, *, argmax=None, raw_scores=None,
                           q_scale: float = 1.0, d_scale: float = 1.0, stream=None):
    """C: ``maxsim_forward_noalloc`` -- maxsim_forward for callers that cannot
    allocate device memory: the scratch lives in a fixed array owned by the
    library, so only caller-provided outputs are written (``scores`` and the
    optional ``argmax`` / ``raw_scores`` must be passed in).  Calls that
    overlap on the GPU share that array and must be serialised."""
    torch = _torch()
    lib = load_library()
    _check_qd(Q, D)
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    # the outputs are written without bounds checks: their shapes, dtypes and
    # device are checked first, before anything reaches the library
    _check_forward_outputs(n_q, n_docs, lq_max, Q.device, scores, argmax, raw_scores)
    if raw_scores is not None and Q.dtype != torch.int8:
        raise ValueError("raw_scores is an INT8 output")
    _require(Q, "Q")
    dev = Q.device
    _require(D, "D", dtype=Q.dtype, device=dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if q_lens.shape != (n_q,):
        raise ValueError(f"q_lens must have shape ({n_q},)")
    with torch.cuda.device(dev):
        st = lib.maxsim_forward_noalloc(_ptr(Q), _ptr(q_lens), n_q, lq_max, _ptr(D), _ptr(cu_seqlens),
                                        n_docs, D.shape[0], dim, _dtype_code(Q),
                                        float(q_scale), float(d_scale), _ptr(scores), _ptr(raw_scores),
                                        _ptr(argmax), _stream(stream))
    _check("maxsim_forward_noalloc", st)
    return scores, argmax, raw_scores


def maxsim_forward_host_workspace_size(n_q: int, lq_max: int, n_docs: int, block_docs: int, block_tokens: int,
                                       dtype, dim: int = 128) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return int(load_library().maxsim_forward_host_workspace_size(n_q, lq_max, n_docs, block_docs, block_tokens,
                                                                 dim, code))


_COPY_STREAMS = {}


def _copy_stream_for(dev):
    torch = _torch()
    if dev not in _COPY_STREAMS:
        _COPY_STREAMS[dev] = torch.cuda.Stream(device=dev)
    return _COPY_STREAMS[dev]


def maxsim_forward_host(Q, q_lens, D_host, cu_seqlens_host, *, block_docs: int, block_tokens: int = None,
                        with_argmax: bool = False, q_scale: float = 1.0, d_scale: float = 1.0, scores=None,
                        argmax=None, raw_scores=None, want_raw: bool = False, workspace=None,
                        overlap: bool = True, copy_stream=None, stream=None):
    """C: ``maxsim_forward_host`` -- out-of-core scoring: Q and q_lens on the
    device, the corpus (D_host [total, 128], cu_seqlens_host [n_docs+1]
    int32) in host memory.  Blocks of consecutive documents (at most
    ``block_docs`` documents and ``block_tokens`` tokens) are copied to the
    device on ``copy_stream`` (a cached side stream by default; the compute
    stream when ``overlap`` is False) and scored while the next block is
    copied.  D_host should be pinned (``tensor.pin_memory()``) for the
    copies to overlap, and must stay alive and unchanged until ``stream``
    has synchronised.  Returns device tensors like ``maxsim_forward``."""
    torch = _torch()
    lib = load_library()
    _require(Q, "Q")
    dev = Q.device
    _require(q_lens, "q_lens", torch.int32, dev)
    if not isinstance(D_host, torch.Tensor) or D_host.is_cuda or not D_host.is_contiguous():
        raise ValueError("D_host must be a contiguous host tensor")
    if D_host.dtype != Q.dtype:
        raise TypeError(f"D_host must be {Q.dtype}, got {D_host.dtype}")
    if (not isinstance(cu_seqlens_host, torch.Tensor) or cu_seqlens_host.is_cuda
            or cu_seqlens_host.dtype != torch.int32 or not cu_seqlens_host.is_contiguous()):
        raise ValueError("cu_seqlens_host must be a contiguous int32 host tensor")
    if Q.dim() != 3 or D_host.dim() != 2 or Q.shape[2] != D_host.shape[1]:
        raise ValueError("Q must be [n_q, lq_max, dim] and D_host [total, dim]")
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens_host.numel() - 1
    total = D_host.shape[0]
    code = _dtype_code(Q)
    if block_tokens is None:
        lens = cu_seqlens_host[1:] - cu_seqlens_host[:-1]
        longest = int(lens.max()) if n_docs > 0 else 1
        block_tokens = max(1, longest) * block_docs
    if scores is None:
        scores = torch.empty((n_q, n_docs), dtype=torch.float32, device=dev)
    if with_argmax and argmax is None:
        argmax = torch.empty((n_q, n_docs, lq_max), dtype=torch.int32, device=dev)
    if not with_argmax:
        argmax = None
    if code == 2 and want_raw and raw_scores is None:
        raw_scores = torch.empty((n_q, n_docs), dtype=torch.int64, device=dev)
    ws_bytes = maxsim_forward_host_workspace_size(n_q, lq_max, n_docs, block_docs, block_tokens, code, dim)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    if overlap and copy_stream is None:
        copy_stream = _copy_stream_for(dev)
    cs = ctypes.c_void_p(copy_stream.cuda_stream) if overlap else None
    with torch.cuda.device(dev):
        st = lib.maxsim_forward_host(_ptr(Q), _ptr(q_lens), n_q, lq_max, ctypes.c_void_p(D_host.data_ptr()),
                                     ctypes.c_void_p(cu_seqlens_host.data_ptr()), n_docs, total, dim, code,
                                     float(q_scale), float(d_scale), _ptr(scores), _ptr(raw_scores),
                                     _ptr(argmax), int(block_docs), int(block_tokens), _ptr(workspace),
                                     workspace.numel(), _stream(stream), cs)
    _check("maxsim_forward_host", st)
    return scores, argmax, raw_scores


def maxsim_forward_int8_per_token(Q, q_scales, q_lens, D, d_scales, cu_seqlens, *, with_argmax: bool = True,
                                  scores=None, argmax=None, workspace=None, stream=None):
    """C: ``maxsim_forward_int8_per_token`` -- INT8 MaxSim with one scale
    per token: Q int8 [n_q, lq_max, 128] with q_scales float32 [n_q,
    lq_max]; D int8 [total, 128] with d_scales float32 [total].  Returns
    (scores [n_q, n_docs] float32, argmax or None)."""
    torch = _torch()
    lib = load_library()
    _require(Q, "Q", torch.int8)
    dev = Q.device
    _require(D, "D", torch.int8, dev)
    _require(q_scales, "q_scales", torch.float32, dev)
    _require(d_scales, "d_scales", torch.float32, dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    if q_scales.shape != (n_q, lq_max) or d_scales.shape != (D.shape[0],):
        raise ValueError("q_scales must be [n_q, lq_max] and d_scales [total]")
    if scores is None:
        scores = torch.empty((n_q, n_docs), dtype=torch.float32, device=dev)
    if with_argmax and argmax is None:
        argmax = torch.empty((n_q, n_docs, lq_max), dtype=torch.int32, device=dev)
    if not with_argmax:
        argmax = None
    ws_bytes = maxsim_forward_workspace_size(n_q, lq_max, n_docs, 2, dim)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_forward_int8_per_token(_ptr(Q), _ptr(q_scales), _ptr(q_lens), n_q, lq_max, _ptr(D),
                                               _ptr(d_scales), _ptr(cu_seqlens), n_docs, D.shape[0], dim,
                                               _ptr(scores), _ptr(argmax), _ptr(workspace),
                                               workspace.numel() if workspace is not None else 0,
                                               _stream(stream))
    _check("maxsim_forward_int8_per_token", st)
    return scores, argmax


def maxsim_topk(values, k: int, *, out_ids=None, out_values=None, stream=None):
    """C: ``maxsim_topk`` -- per row of values [n_rows, n_cols] (float32,
    CUDA; rows may be strided), the k largest entries, descending, ties to
    the lower column.  Returns (ids int32 [n_rows, k], values [n_rows, k])."""
    torch = _torch()
    lib = load_library()
    if values.dim() != 2 or values.dtype != torch.float32 or not values.is_cuda or values.stride(1) != 1:
        raise ValueError("values must be a float32 CUDA matrix with unit column stride")
    n_rows, n_cols = values.shape
    dev = values.device
    if out_ids is None:
        out_ids = torch.empty((n_rows, k), dtype=torch.int32, device=dev)
    if out_values is None:
        out_values = torch.empty((n_rows, k), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_topk(_ptr(values), n_rows, n_cols, values.stride(0) if n_rows > 1 else n_cols, k,
                             _ptr(out_ids), _ptr(out_values), _stream(stream))
    _check("maxsim_topk", st)
    return out_ids, out_values


def maxsim_rerank_workspace_size(n_q: int, lq_max: int, n_docs: int, k_candidates: int, max_doc_len: int,
                                 dtype16, dim: int = 128) -> int:
    code = DTYPE_CODES[dtype16] if isinstance(dtype16, str) else int(dtype16)
    return int(load_library().maxsim_rerank_workspace_size(n_q, lq_max, n_docs, k_candidates, max_doc_len, dim,
                                                           code))


def maxsim_rerank_two_stage(Q8, D8, Q16, D16, q_lens, cu_seqlens, *, k_candidates: int, k: int,
                            q_scale: float = 1.0, d_scale: float = 1.0, q_tok_scales=None, d_tok_scales=None,
                            max_doc_len: int = None, workspace=None, return_candidates: bool = False,
                            stream=None):
    """C: ``maxsim_rerank_two_stage`` -- INT8 scan of every document, the
    k_candidates best per query rescored with the FP16/BF16 tokens, the k
    best returned.  D16 may be a CUDA tensor or a pinned host tensor (the
    gather then reads the candidates' rows over the host link).  Returns
    (ids int32 [n_q, k], scores float32 [n_q, k], candidate ids or None)."""
    torch = _torch()
    lib = load_library()
    _require(Q8, "Q8", torch.int8)
    dev = Q8.device
    _require(D8, "D8", torch.int8, dev)
    _require(Q16, "Q16", None, dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if D16.is_cuda:
        _require(D16, "D16", Q16.dtype, dev)
    elif not (D16.is_pinned() and D16.is_contiguous() and D16.dtype == Q16.dtype):
        raise ValueError("a host D16 must be a contiguous pinned tensor of Q16's dtype")
    n_q, lq_max, dim = Q8.shape
    n_docs = cu_seqlens.numel() - 1
    code16 = _dtype_code(Q16)
    if max_doc_len is None:
        max_doc_len = int((cu_seqlens[1:] - cu_seqlens[:-1]).max()) if n_docs else 0
    ws_bytes = maxsim_rerank_workspace_size(n_q, lq_max, n_docs, k_candidates, max_doc_len, code16, dim)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=dev)
    ids = torch.empty((n_q, k), dtype=torch.int32, device=dev)
    scores = torch.empty((n_q, k), dtype=torch.float32, device=dev)
    cand = torch.empty((n_q, k_candidates), dtype=torch.int32, device=dev) if return_candidates else None
    with torch.cuda.device(dev):
        st = lib.maxsim_rerank_two_stage(
            _ptr(Q8), _ptr(q_tok_scales), float(q_scale), _ptr(D8), _ptr(d_tok_scales), float(d_scale),
            _ptr(Q16), ctypes.c_void_p(D16.data_ptr()), code16, _ptr(q_lens), n_q, lq_max, _ptr(cu_seqlens),
            n_docs, D8.shape[0], max_doc_len, dim, k_candidates, k, _ptr(ids), _ptr(scores), _ptr(cand),
            _ptr(workspace), workspace.numel(), _stream(stream))
    _check("maxsim_rerank_two_stage", st)
    return ids, scores, cand


def _sets(P, cu_p, Q, cu_q):
    torch = _torch()
    _require(P, "P", torch.float32)
    dev = P.device
    _require(Q, "Q", torch.float32, dev)
    _require(cu_p, "cu_p", torch.int32, dev)
    _require(cu_q, "cu_q", torch.int32, dev)
    if P.dim() != 2 or P.shape[1] != 3 or Q.dim() != 2 or Q.shape[1] != 3:
        raise ValueError("P and Q must be [total, 3] float32")
    if cu_p.numel() != cu_q.numel():
        raise ValueError("cu_p and cu_q must describe the same number of items")
    return dev


def maxsim_chamfer_forward(P, cu_p, Q, cu_q, *, max_p: int = None, max_q: int = None, workspace=None,
                           stream=None):
    """C: ``maxsim_chamfer_forward`` -- Chamfer distance of each item of a
    packed batch of point-set pairs.  Returns (cd [B] float32, dist_pq,
    arg_pq, dist_qp, arg_qp)."""
    torch = _torch()
    lib = load_library()
    dev = _sets(P, cu_p, Q, cu_q)
    n_items = cu_p.numel() - 1
    if max_p is None:
        max_p = int((cu_p[1:] - cu_p[:-1]).max()) if n_items else 0
    if max_q is None:
        max_q = int((cu_q[1:] - cu_q[:-1]).max()) if n_items else 0
    N, M = P.shape[0], Q.shape[0]
    cd = torch.empty(n_items, dtype=torch.float32, device=dev)
    d_pq = torch.empty(N, dtype=torch.float32, device=dev)
    a_pq = torch.empty(N, dtype=torch.int32, device=dev)
    d_qp = torch.empty(M, dtype=torch.float32, device=dev)
    a_qp = torch.empty(M, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        ws_bytes = int(lib.maxsim_chamfer_forward_workspace_size(n_items, N, M, max_p, max_q))
        if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        st = lib.maxsim_chamfer_forward(_ptr(P), _ptr(cu_p), _ptr(Q), _ptr(cu_q), n_items, N, M, max_p, max_q,
                                        _ptr(cd), _ptr(d_pq), _ptr(a_pq), _ptr(d_qp), _ptr(a_qp), _ptr(workspace),
                                        workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("maxsim_chamfer_forward", st)
    return cd, d_pq, a_pq, d_qp, a_qp


def maxsim_chamfer_build_csr(arg, cu_src, cu_dst, total_dst: int, *, workspace=None, stream=None):
    """C: ``maxsim_chamfer_build_csr`` -- (row_ptr [total_dst + 1], col_idx
    [n_sources]) of a nearest-neighbour map; col_idx[:row_ptr[-1]] is valid."""
    torch = _torch()
    lib = load_library()
    _require(arg, "arg", torch.int32)
    dev = arg.device
    n_items = cu_src.numel() - 1
    row_ptr = torch.empty(total_dst + 1, dtype=torch.int32, device=dev)
    col = torch.empty(max(arg.numel(), 1), dtype=torch.int32, device=dev)
    need = int(lib.maxsim_chamfer_csr_workspace_size(arg.numel(), total_dst))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_chamfer_build_csr(_ptr(arg), _ptr(cu_src), _ptr(cu_dst), n_items, arg.numel(), total_dst,
                                          _ptr(row_ptr), _ptr(col), _ptr(workspace), workspace.numel(),
                                          _stream(stream))
    _check("maxsim_chamfer_build_csr", st)
    return row_ptr, col[:arg.numel()]


def maxsim_chamfer_backward(grad_cd, P, cu_p, Q, cu_q, arg_pq, arg_qp, *, workspace=None, stream=None):
    """C: ``maxsim_chamfer_backward`` -- (dP [N, 3], dQ [M, 3]) float32 of
    sum_b grad_cd[b] * CD_b through the saved nearest-neighbour indices."""
    torch = _torch()
    lib = load_library()
    dev = _sets(P, cu_p, Q, cu_q)
    _require(grad_cd, "grad_cd", torch.float32, dev)
    n_items = cu_p.numel() - 1
    N, M = P.shape[0], Q.shape[0]
    dP = torch.empty((N, 3), dtype=torch.float32, device=dev)
    dQ = torch.empty((M, 3), dtype=torch.float32, device=dev)
    need = int(lib.maxsim_chamfer_backward_workspace_size(N, M))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_chamfer_backward(_ptr(grad_cd), _ptr(P), _ptr(cu_p), _ptr(Q), _ptr(cu_q), n_items, N, M,
                                         _ptr(arg_pq), _ptr(arg_qp), _ptr(dP), _ptr(dQ), _ptr(workspace),
                                         workspace.numel(), _stream(stream))
    _check("maxsim_chamfer_backward", st)
    return dP, dQ


def maxsim_build_csr(argmax, q_lens, cu_seqlens, total_d_tokens: int, *, workspace=None, stream=None):
    """Inverse-grid CSR of an argmax map (C: ``maxsim_build_csr``).
    Returns (row_ptr [total+1] int32, col_idx [n_sources] int32)."""
    torch = _torch()
    lib = load_library()
    _require(argmax, "argmax", torch.int32)
    dev = argmax.device
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_q, n_docs, lq_max = argmax.shape
    row_ptr = torch.empty(total_d_tokens + 1, dtype=torch.int32, device=dev)
    col_idx = torch.empty(max(1, n_q * n_docs * lq_max), dtype=torch.int32, device=dev)
    ws_bytes = maxsim_backward_workspace_size(n_q, lq_max, n_docs, total_d_tokens)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_build_csr(_ptr(argmax), _ptr(q_lens), n_q, lq_max, _ptr(cu_seqlens), n_docs,
                                  total_d_tokens, _ptr(row_ptr), _ptr(col_idx), _ptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check("maxsim_build_csr", st)
    nnz = int(row_ptr[-1].item())
    return row_ptr, col_idx[:nnz]


def maxsim_backward(grad_scores, argmax, Q, q_lens, D, cu_seqlens, *, dQ=None, dD=None,
                    workspace=None, stream=None):
    """Backward of the fused MaxSim (C: ``maxsim_backward``).
    Returns (dQ [n_q, lq_max, 128] float32, dD [total, 128] float32)."""
    torch = _torch()
    lib = load_library()
    _require(Q, "Q")
    dev = Q.device
    _require(D, "D", dtype=Q.dtype, device=dev)
    _require(grad_scores, "grad_scores", torch.float32, dev)
    _require(argmax, "argmax", torch.int32, dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    total = D.shape[0]
    if dQ is None:
        dQ = torch.empty((n_q, lq_max, dim), dtype=torch.float32, device=dev)
    if dD is None:
        dD = torch.empty((total, dim), dtype=torch.float32, device=dev)
    ws_bytes = maxsim_backward_workspace_size(n_q, lq_max, n_docs, total)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_backward(_ptr(grad_scores), _ptr(argmax), _ptr(Q), _ptr(q_lens), n_q, lq_max,
                                 _ptr(D), _ptr(cu_seqlens), n_docs, total, dim, _dtype_code(Q),
                                 _ptr(dQ), _ptr(dD), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check("maxsim_backward", st)
    return dQ, dD


def maxsim_forward_with_counts(Q, q_lens, D, cu_seqlens, *, scores=None, argmax=None, workspace=None,
                               backward_workspace=None, stream=None):
    """C: ``maxsim_forward_with_counts`` -- the training forward (FP16/BF16):
    scores and argmax as ``maxsim_forward`` (nothing is counted any more: the
    backward sorts each document's sources itself).  Returns (scores, argmax,
    backward_workspace); pass the last two to ``maxsim_backward_with_counts``."""
    torch = _torch()
    lib = load_library()
    _require(Q, "Q")
    dev = Q.device
    _require(D, "D", dtype=Q.dtype, device=dev)
    _require(q_lens, "q_lens", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    total = D.shape[0]
    code = _dtype_code(Q)
    if scores is None:
        scores = torch.empty((n_q, n_docs), dtype=torch.float32, device=dev)
    if argmax is None:
        argmax = torch.empty((n_q, n_docs, lq_max), dtype=torch.int32, device=dev)
    ws_bytes = maxsim_forward_workspace_size(n_q, lq_max, n_docs, code, dim)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    bws_bytes = maxsim_backward_workspace_size(n_q, lq_max, n_docs, total)
    if backward_workspace is None or backward_workspace.numel() < bws_bytes:
        backward_workspace = torch.empty(max(bws_bytes, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_forward_with_counts(_ptr(Q), _ptr(q_lens), n_q, lq_max, _ptr(D), _ptr(cu_seqlens), n_docs,
                                            total, dim, code, _ptr(scores), _ptr(argmax), _ptr(workspace),
                                            workspace.numel() if workspace is not None else 0,
                                            _ptr(backward_workspace), backward_workspace.numel(), _stream(stream))
    _check("maxsim_forward_with_counts", st)
    return scores, argmax, backward_workspace


def maxsim_backward_with_counts(grad_scores, argmax, Q, q_lens, D, cu_seqlens, backward_workspace, *, dQ=None,
                                dD=None, stream=None):
    """C: ``maxsim_backward_with_counts`` -- ``maxsim_backward`` with the
    workspace ``maxsim_forward_with_counts`` returned.  Returns (dQ, dD)
    float32."""
    torch = _torch()
    lib = load_library()
    _require(grad_scores, "grad_scores", torch.float32)
    dev = grad_scores.device
    n_q, lq_max, dim = Q.shape
    n_docs = cu_seqlens.numel() - 1
    total = D.shape[0]
    if dQ is None:
        dQ = torch.empty((n_q, lq_max, dim), dtype=torch.float32, device=dev)
    if dD is None:
        dD = torch.empty((total, dim), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib.maxsim_backward_with_counts(_ptr(grad_scores), _ptr(argmax), _ptr(Q), _ptr(q_lens), n_q, lq_max,
                                             _ptr(D), _ptr(cu_seqlens), n_docs, total, dim, _dtype_code(Q),
                                             _ptr(dQ), _ptr(dD), _ptr(backward_workspace),
                                             backward_workspace.numel(), _stream(stream))
    _check("maxsim_backward_with_counts", st)
    return dQ, dD


def maxsim_forward_plan(n_q: int, lq_max: int, n_docs: int, total_d_tokens: int, dtype="fp16", *,
                        with_argmax: bool = True, sm_count: int | None = None) -> dict:
    """C: ``maxsim_forward_plan`` -- the forward's launch layout for these
    sizes (host only).  ``dtype`` is "fp16", "bf16" or "int8" (or a torch
    dtype); ``sm_count`` defaults to the current CUDA device's."""
    lib = load_library()
    if sm_count is None:
        torch = _torch()
        sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if not isinstance(dtype, str):
        torch = _torch()
        dtype = {torch.float16: "fp16", torch.bfloat16: "bf16", torch.int8: "int8"}[dtype]
    code = DTYPE_CODES[dtype]
    out = (ctypes.c_int32 * 5)()
    _check("maxsim_forward_plan", lib.maxsim_forward_plan(int(n_q), int(lq_max), int(n_docs), int(total_d_tokens),
                                                          code, 1 if with_argmax else 0, int(sm_count), out))
    return {"m_tiles": out[0], "ctas_per_sm": out[1], "row_groups": out[2], "parts": out[3],
            "k_block_halves": bool(out[4])}


PROBE_SINK_WORDS = 1024


def maxsim_probe_l2_read(buf, passes: int, sink=None, stream=None):
    """C: ``maxsim_probe_l2_read`` -- enqueue ``passes`` plain reads of the
    device buffer ``buf`` (contiguous, 16-byte aligned, a multiple of 16
    bytes); time them with events on ``stream``.  Returns the sink tensor
    (uint64 words as int64 [1024])."""
    torch = _torch()
    lib = load_library()
    _require(buf, "buf")
    if sink is None:
        sink = torch.zeros(PROBE_SINK_WORDS, dtype=torch.int64, device=buf.device)
    _check_output(sink, "sink", (PROBE_SINK_WORDS,), torch.int64, buf.device)
    nbytes = buf.numel() * buf.element_size()
    with torch.cuda.device(buf.device):
        st = lib.maxsim_probe_l2_read(_ptr(buf), nbytes, int(passes), _ptr(sink), _stream(stream))
    _check("maxsim_probe_l2_read", st)
    return sink


def maxsim_selftest_bounded_wait(limit_us: int = 5000, stream=None) -> None:
    """C: ``maxsim_selftest_bounded_wait`` -- enqueue the bounded-wait
    self-test (one CTA whose wait gives up after ``limit_us`` microseconds and
    records 0x105 in the device status word)."""
    lib = load_library()
    _check("maxsim_selftest_bounded_wait", lib.maxsim_selftest_bounded_wait(int(limit_us), _stream(stream)))


def maxsim_device_status(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device status word (0 = ok)."""
    lib = load_library()
    code = ctypes.c_int32(0)
    st = lib.maxsim_device_status(_stream(stream), 1 if clear else 0, ctypes.byref(code))
    if st not in (0, 5):
        _check("maxsim_device_status", st)
    return int(code.value)
