"""Sparse embedding weight-gradient accumulation on GB300 (sm_103a).

``accumulate_embedding_wgrad(ids, grad, main_grad)`` performs
``main_grad += embedding_dense_backward(grad, ids)`` touching only the rows of the ids
that occur, with the values of PyTorch's sort-based embedding backward followed by
``main_grad.add_`` (Megatron Core API docs, ``core.fusions.fused_embedding_wgrad``:
module docstring, ``accumulate_embedding_wgrad`` and ``can_accumulate_embedding_wgrad``).

This module only marshals arguments into the C ABI of ``libewg.so`` (declared in
``include/ewg.h``); every step of the computation runs in that library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no CPU
fallback: without the compiled library every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "MIN_TOKENS", "MAX_TOKENS", "NROWS", "EwgError", "can_accumulate_embedding_wgrad",
    "accumulate_embedding_wgrad", "workspace_bytes", "plan", "apply", "read_status",
    "library_path", "lib", "accumulate_embedding_wgrad_shard",
]

MIN_TOKENS = 3073
MAX_TOKENS = 1 << 28
NROWS = 10

_INT32, _INT64, _BF16, _FP32 = 0, 1, 2, 3
OK, ERR_UNSUPPORTED, ERR_INVALID, ERR_CUDA, ERR_ID_OUT_OF_RANGE, ERR_TIMEOUT, ERR_BOUNDS = \
    0, 1, 2, 3, 4, 5, 6

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libewg.so")
# The same library built with every kernel index checked (EWG_ERR_BOUNDS on a failure).
_DEBUG_LIB_PATH = os.path.join(_HERE, "libewg_debug.so")
_lib = None
_debug_lib = None
_lock = threading.Lock()
# Pinned host tensors handed to the host-input call, each kept alive until an event
# recorded after the call has completed: the library copies from their raw pointers, so
# torch's pinned-memory allocator does not know the copies are still pending.
_pending_host = []
_pending_lock = threading.Lock()


class EwgError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded C library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _load(_LIB_PATH)
    return _lib


def debug_lib():
    """The bounds-checking build of the same library (libewg_debug.so), for tests."""
    global _debug_lib
    if _debug_lib is not None:
        return _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _load(_DEBUG_LIB_PATH)
    return _debug_lib


def _load(path):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m embedding_weight_grad_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    L.ewg_can_accumulate.argtypes = [vp, i32, i64, vp, i32, i64, vp, i32, i64, i64, i64]
    L.ewg_can_accumulate.restype = i32
    L.ewg_workspace_bytes.argtypes = [i64, i64]
    L.ewg_workspace_bytes.restype = sz
    L.ewg_accumulate.argtypes = [vp, i32, i64, vp, i32, i64, vp, i32, i64, i64, i64, vp,
                                 sz, vp]
    L.ewg_accumulate.restype = i32
    L.ewg_plan.argtypes = [vp, i32, i64, i64, i64, vp, sz, vp]
    L.ewg_plan.restype = i32
    L.ewg_apply.argtypes = [vp, i32, i64, vp, i32, i64, i64, i64, i64, vp, sz, vp]
    L.ewg_apply.restype = i32
    L.ewg_accumulate_shard.argtypes = [vp, i32, i64, vp, i32, i64, vp, i32, i64, i64, i64,
                                       i64, i64, vp, sz, vp]
    L.ewg_accumulate_shard.restype = i32
    L.ewg_plan_shard.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, sz, vp]
    L.ewg_plan_shard.restype = i32
    L.ewg_host_workspace_bytes.argtypes = [i64, i64, i32, i32]
    L.ewg_host_workspace_bytes.restype = sz
    L.ewg_accumulate_host.argtypes = [vp, i32, i64, vp, i32, vp, i32, i64, i64, i64, vp,
                                      sz, vp]
    L.ewg_accumulate_host.restype = i32
    L.ewg_read_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    L.ewg_read_status.restype = i32
    L.ewg_status_string.argtypes = [i32]
    L.ewg_status_string.restype = ctypes.c_char_p
    L.ewg_last_error.argtypes = []
    L.ewg_last_error.restype = ctypes.c_char_p
    L.ewg_version.argtypes = []
    L.ewg_version.restype = i32
    return L


def _raise_on(code: int):
    if code != OK:
        L = lib()
        raise EwgError(code, f"{L.ewg_status_string(code).decode()}: {L.ewg_last_error().decode()}")


_FLOAT_CODES = {torch.bfloat16: _BF16, torch.float32: _FP32}
_ID_CODES = {torch.int32: _INT32, torch.int64: _INT64}


def _stream_ptr(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class _Args:
    """The C-ABI view of (ids, grad, main_grad), or the reason there is none."""

    def __init__(self, ids: torch.Tensor, grad: torch.Tensor, main_grad: torch.Tensor):
        self.reason = None
        if not (ids.is_cuda and grad.is_cuda and main_grad.is_cuda):
            self.reason = "tensors must be on a CUDA device"
            return
        if ids.dtype not in _ID_CODES or grad.dtype not in _FLOAT_CODES \
                or main_grad.dtype not in _FLOAT_CODES:
            self.reason = "ids must be int32/int64; grad and main_grad bf16/fp32"
            return
        if main_grad.dim() != 2 or main_grad.stride(1) != 1:
            self.reason = "main_grad must be [num_embeddings, hidden] with unit inner stride"
            return
        if not ids.is_contiguous():
            self.reason = "ids must be contiguous"
            return
        V, H = main_grad.shape
        n = ids.numel()
        if tuple(grad.shape) != tuple(ids.shape) + (H,):
            self.reason = "grad must be [*ids.shape, hidden]"
            return
        try:
            g2 = grad.view(n, H)
        except RuntimeError:
            self.reason = "grad rows must share one row stride"
            return
        if H > 0 and n > 0 and g2.stride(1) != 1:
            self.reason = "grad must have unit inner stride"
            return
        self.ids, self.grad, self.main_grad = ids.reshape(n), g2, main_grad
        self.n, self.V, self.H = n, V, H
        self.grad_stride = g2.stride(0) if n > 1 else H
        self.mg_stride = main_grad.stride(0) if V > 1 else H
        self.device = main_grad.device

    def c_args(self):
        return (self.ids.data_ptr(), _ID_CODES[self.ids.dtype], self.n,
                self.grad.data_ptr(), _FLOAT_CODES[self.grad.dtype], self.grad_stride,
                self.main_grad.data_ptr(), _FLOAT_CODES[self.main_grad.dtype], self.V, self.H,
                self.mg_stride)


def can_accumulate_embedding_wgrad(ids: torch.Tensor, grad: torch.Tensor,
                                   main_grad: torch.Tensor) -> bool:
    """Whether accumulate_embedding_wgrad supports these tensors (see include/ewg.h)."""
    a = _Args(ids, grad, main_grad)
    if a.reason is not None:
        return False
    with torch.cuda.device(a.device):
        return bool(lib().ewg_can_accumulate(*a.c_args()))


def workspace_bytes(num_tokens: int, hidden: int) -> int:
    return int(lib().ewg_workspace_bytes(num_tokens, hidden))


def new_workspace(num_tokens: int, hidden: int, device=None) -> torch.Tensor:
    """A device buffer large enough for any call with these sizes (no init needed)."""
    nbytes = workspace_bytes(num_tokens, hidden)
    if nbytes == 0:
        raise EwgError(ERR_UNSUPPORTED, "unsupported num_tokens / hidden")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def accumulate_embedding_wgrad(ids: torch.Tensor, grad: torch.Tensor, main_grad: torch.Tensor,
                               *, workspace: torch.Tensor | None = None,
                               check: bool = False) -> None:
    """main_grad += embedding_dense_backward(grad, ids), touching only the rows of ids.

    ids: token ids, any shape, num_tokens elements; grad: [*ids.shape, hidden];
    main_grad: [num_embeddings, hidden], updated in place.  Requires
    can_accumulate_embedding_wgrad(ids, grad, main_grad) (raises ValueError otherwise).
    The work is enqueued on the current stream.  With check=True the call waits for it
    and raises EwgError if the device found an id outside [0, num_embeddings), in which
    case main_grad was left untouched.
    """
    a = _Args(ids, grad, main_grad)
    if a.reason is not None:
        raise ValueError(f"accumulate_embedding_wgrad does not support these tensors: {a.reason}")
    with torch.cuda.device(a.device):
        L = lib()
        if not L.ewg_can_accumulate(*a.c_args()):
            raise ValueError("accumulate_embedding_wgrad does not support these tensors: "
                             + L.ewg_last_error().decode())
        ws = workspace if workspace is not None else new_workspace(a.n, a.H, a.device)
        stream = _stream_ptr(a.device)
        _raise_on(L.ewg_accumulate(*a.c_args(), ws.data_ptr(), ws.numel(), stream))
        if check:
            raise_on_device_status(ws)


def new_host_workspace(num_tokens: int, hidden: int, ids_dtype: torch.dtype,
                       grad_dtype: torch.dtype, device=None) -> torch.Tensor:
    """A device buffer for accumulate_embedding_wgrad_from_host with these sizes and dtypes."""
    nbytes = int(lib().ewg_host_workspace_bytes(num_tokens, hidden, _ID_CODES.get(ids_dtype, -1),
                                                _FLOAT_CODES.get(grad_dtype, -1)))
    if nbytes == 0:
        raise EwgError(ERR_UNSUPPORTED, "unsupported num_tokens / hidden / dtypes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _keep_until_passed(stream, tensors) -> None:
    """Holds `tensors` until `stream` has passed the work enqueued so far; entries whose
    event has completed are dropped on every call."""
    ev = torch.cuda.Event()
    ev.record(stream)
    with _pending_lock:
        _pending_host[:] = [(e, t) for (e, t) in _pending_host if not e.query()]
        _pending_host.append((ev, tensors))


def accumulate_embedding_wgrad_from_host(ids: torch.Tensor, grad: torch.Tensor,
                                         main_grad: torch.Tensor, *,
                                         workspace: torch.Tensor | None = None,
                                         check: bool = False) -> None:
    """accumulate_embedding_wgrad with ids and grad in pinned host memory: the library
    copies them to the device (the grad copy overlapping the plan) and accumulates into
    main_grad on its device, all enqueued on the current stream.  ids: contiguous CPU
    int32/int64 tensor, grad: contiguous CPU bf16/fp32 tensor [*ids.shape, hidden], both
    pinned; main_grad: CUDA [num_embeddings, hidden].  check=True as in
    accumulate_embedding_wgrad.

    The copies run after the call returns.  This function keeps ids and grad alive until
    the stream has passed the call, so dropping them (or a temporary ``x.pin_memory()``)
    right away is safe; writing new values into them before the stream has passed the
    call is not (synchronize the stream, or wait on an event recorded after the call)."""
    if ids.is_cuda or grad.is_cuda or not main_grad.is_cuda:
        raise ValueError("ids and grad must be host tensors, main_grad a CUDA tensor")
    if not (ids.is_contiguous() and grad.is_contiguous() and ids.is_pinned() and grad.is_pinned()):
        raise ValueError("ids and grad must be contiguous pinned host tensors")
    if ids.dtype not in _ID_CODES or grad.dtype not in _FLOAT_CODES \
            or main_grad.dtype not in _FLOAT_CODES or main_grad.dim() != 2 or main_grad.stride(1) != 1:
        raise ValueError("unsupported dtypes or main_grad layout")
    V, H = main_grad.shape
    n = ids.numel()
    if tuple(grad.shape) != tuple(ids.shape) + (H,):
        raise ValueError("grad must be [*ids.shape, hidden]")
    with torch.cuda.device(main_grad.device):
        L = lib()
        ws = workspace if workspace is not None else new_host_workspace(n, H, ids.dtype, grad.dtype,
                                                                        main_grad.device)
        _raise_on(L.ewg_accumulate_host(
            ids.data_ptr(), _ID_CODES[ids.dtype], n, grad.data_ptr(), _FLOAT_CODES[grad.dtype],
            main_grad.data_ptr(), _FLOAT_CODES[main_grad.dtype], V, H,
            main_grad.stride(0) if V > 1 else H, ws.data_ptr(), ws.numel(),
            _stream_ptr(main_grad.device)))
        _keep_until_passed(torch.cuda.current_stream(main_grad.device), (ids, grad))
        if check:
            raise_on_device_status(ws)


def accumulate_embedding_wgrad_shard(ids: torch.Tensor, grad: torch.Tensor,
                                     main_grad_shard: torch.Tensor, row_begin: int,
                                     num_embeddings: int, *,
                                     workspace: torch.Tensor | None = None,
                                     check: bool = False) -> None:
    """accumulate_embedding_wgrad restricted to the table rows
    [row_begin, row_begin + main_grad_shard.shape[0]) of a num_embeddings-row table.

    main_grad_shard holds those rows (its row 0 is table row row_begin) and ends with
    the bits the whole-table call would give them; ids of other rows are skipped, ids
    outside [0, num_embeddings) are errors.  One GPU per row range needs no exchange.
    """
    a = _Args(ids, grad, main_grad_shard)
    if a.reason is not None:
        raise ValueError(f"accumulate_embedding_wgrad_shard does not support these tensors: {a.reason}")
    rows = a.V
    with torch.cuda.device(a.device):
        L = lib()
        ws = workspace if workspace is not None else new_workspace(a.n, a.H, a.device)
        args = list(a.c_args())
        args[8:9] = [num_embeddings, row_begin, rows]   # V -> (num_embeddings, row_begin, rows)
        _raise_on(L.ewg_accumulate_shard(*args, ws.data_ptr(), ws.numel(), _stream_ptr(a.device)))
        if check:
            raise_on_device_status(ws)


def read_status(workspace: torch.Tensor) -> int:
    """Waits for the current stream and returns the device status of the last call."""
    status = ctypes.c_int(-1)
    with torch.cuda.device(workspace.device):
        _raise_on(lib().ewg_read_status(workspace.data_ptr(), _stream_ptr(workspace.device),
                                        ctypes.byref(status)))
    return status.value


def raise_on_device_status(workspace: torch.Tensor) -> None:
    s = read_status(workspace)
    if s != OK:
        raise EwgError(s, f"device reported {lib().ewg_status_string(s).decode()}")


def plan(ids: torch.Tensor, num_embeddings: int, hidden: int, workspace: torch.Tensor) -> None:
    """Sort + run listing of ids into `workspace` (first half of the accumulation)."""
    ids_flat = ids.reshape(-1)
    if ids.dtype not in _ID_CODES or not ids.is_contiguous():
        raise ValueError("ids must be contiguous int32/int64")
    with torch.cuda.device(ids.device):
        _raise_on(lib().ewg_plan(ids_flat.data_ptr(), _ID_CODES[ids.dtype], ids_flat.numel(),
                                 num_embeddings, hidden, workspace.data_ptr(), workspace.numel(),
                                 _stream_ptr(ids.device)))


def apply(grad: torch.Tensor, main_grad: torch.Tensor, num_tokens: int,
          workspace: torch.Tensor) -> None:
    """Partial sums and the add into main_grad, using the plan in `workspace`."""
    V, H = main_grad.shape
    g2 = grad.view(num_tokens, H)
    with torch.cuda.device(main_grad.device):
        _raise_on(lib().ewg_apply(g2.data_ptr(), _FLOAT_CODES[grad.dtype],
                                  g2.stride(0) if num_tokens > 1 else H, main_grad.data_ptr(),
                                  _FLOAT_CODES[main_grad.dtype], num_tokens, V, H,
                                  main_grad.stride(0) if V > 1 else H, workspace.data_ptr(),
                                  workspace.numel(), _stream_ptr(main_grad.device)))
