"""CPU oracle for sparse embedding weight-gradient accumulation (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline / reference
arm may import this package.  The product library never loads it, and it shares no
code with the CUDA path.

The arithmetic lives in ``ewg_oracle.cpp`` (plain C++17, built with g++ and no
fast-math); this module only compiles it and marshals numpy arrays through ctypes.
bf16 arrays are passed as ``np.uint16`` bit patterns.

Source of the method: Megatron Core API docs, ``core.fusions.fused_embedding_wgrad``,
module docstring (the two bullets on PyTorch's sort-based embedding backward and on
``main_grad.add_``) and the ``accumulate_embedding_wgrad`` entry.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ewg_oracle.cpp")
_LIB = os.path.join(_HERE, "libewg_oracle.so")

INT32, INT64, BF16, FP32 = 0, 1, 2, 3
NROWS = 10

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (g++, IEEE arithmetic)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.ewg_oracle_accumulate.argtypes = [vp, i32, i64, vp, i32, i64, vp, i32, i64,
                                                  i64, i64, i32]
            lib.ewg_oracle_accumulate.restype = i32
            lib.ewg_oracle_weight_grad.argtypes = [vp, i32, i64, vp, i32, i64, i64, i64, vp,
                                                   vp, i32]
            lib.ewg_oracle_weight_grad.restype = i64
            lib.ewg_oracle_sort_pairs.argtypes = [vp, i32, i64, i64, vp, vp]
            lib.ewg_oracle_sort_pairs.restype = i32
            lib.ewg_oracle_round_to_bf16.argtypes = [vp, vp, i64]
            lib.ewg_oracle_round_to_bf16.restype = None
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ids_arg(ids: np.ndarray):
    ids = np.ascontiguousarray(ids).reshape(-1)
    if ids.dtype == np.int64:
        return ids, INT64
    if ids.dtype == np.int32:
        return ids, INT32
    raise TypeError(f"ids must be int32 or int64, got {ids.dtype}")


def _float_arg(a: np.ndarray, name: str):
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return FP32
    raise TypeError(f"{name} must be uint16 (bf16 bits) or float32, got {a.dtype}")


def _rows(a: np.ndarray, name: str):
    """View `a` as [rows, H] with unit inner stride; returns (array, row_stride)."""
    if a.ndim < 2:
        raise ValueError(f"{name} must have a hidden dimension")
    H = a.shape[-1]
    a2 = a.reshape(-1, H) if a.flags.c_contiguous else a
    if a2.ndim != 2 or a2.strides[1] != a2.itemsize:
        a2 = np.ascontiguousarray(a).reshape(-1, H)
    return a2, a2.strides[0] // a2.itemsize


def accumulate(ids: np.ndarray, grad: np.ndarray, main_grad: np.ndarray,
               num_threads: int = 0) -> None:
    """main_grad += embedding_dense_backward(grad, ids), in place, touching only rows of ids.

    ids: any shape, int32/int64; grad: [*ids.shape, H] (uint16 bf16 bits or float32),
    the last dim unit-strided; main_grad: [V, H] (uint16 bf16 bits or float32),
    unit inner stride, modified in place.
    """
    lib = _load()
    ids_flat, ids_dt = _ids_arg(ids)
    n = ids_flat.size
    g_dt = _float_arg(grad, "grad")
    m_dt = _float_arg(main_grad, "main_grad")
    if main_grad.ndim != 2 or main_grad.strides[1] != main_grad.itemsize:
        raise ValueError("main_grad must be [V, H] with unit inner stride")
    V, H = main_grad.shape
    if grad.shape[-1] != H or grad.size // H != n:
        raise ValueError("grad must be [*ids.shape, H]")
    g2, g_stride = _rows(grad, "grad")
    m_stride = main_grad.strides[0] // main_grad.itemsize
    rc = lib.ewg_oracle_accumulate(ids_flat.ctypes.data, ids_dt, n, g2.ctypes.data, g_dt,
                                   g_stride, main_grad.ctypes.data, m_dt, V, H, m_stride,
                                   num_threads)
    if rc != 0:
        raise OracleError(f"oracle accumulate failed with code {rc}")


def weight_grad(ids: np.ndarray, grad: np.ndarray, num_embeddings: int,
                num_threads: int = 0):
    """Rows of embedding_dense_backward(grad, ids) for the ids that occur.

    Returns (uniq_ids int64 [U] ascending, w float32 [U, H]); w holds the values after
    the single rounding to grad's dtype, widened to float32.
    """
    lib = _load()
    ids_flat, ids_dt = _ids_arg(ids)
    n = ids_flat.size
    g_dt = _float_arg(grad, "grad")
    H = grad.shape[-1]
    g2, g_stride = _rows(grad, "grad")
    uniq = np.empty(max(n, 1), dtype=np.int64)
    w = np.empty((max(n, 1), H), dtype=np.float32)
    U = lib.ewg_oracle_weight_grad(ids_flat.ctypes.data, ids_dt, n, g2.ctypes.data, g_dt,
                                   g_stride, num_embeddings, H, uniq.ctypes.data,
                                   w.ctypes.data, num_threads)
    if U < 0:
        raise OracleError(f"oracle weight_grad failed with code {-U}")
    return uniq[:U].copy(), w[:U].copy()


def sort_pairs(ids: np.ndarray, num_embeddings: int):
    """(sorted_ids, sorted_positions), both int64 [n]: step 1 on its own."""
    lib = _load()
    ids_flat, ids_dt = _ids_arg(ids)
    n = ids_flat.size
    sid = np.empty(n, dtype=np.int64)
    spos = np.empty(n, dtype=np.int64)
    rc = lib.ewg_oracle_sort_pairs(ids_flat.ctypes.data, ids_dt, n, num_embeddings,
                                   sid.ctypes.data, spos.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle sort failed with code {rc}")
    return sid, spos


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.ewg_oracle_round_to_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
