"""The allocation-free entry point (ewg_accumulate_static) against ewg_accumulate.

ewg_accumulate_static serves callers that cannot allocate device memory at the time
of the call: it uses a fixed array the library keeps in device memory as its workspace.
This file runs last (its name sorts last) so that a failure here comes after every
other test has run; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
_INT64, _BF16, _FP32 = 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from embedding_weight_grad_gb300 import build
    build.build()
    L = ewg.lib()
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    L.ewg_accumulate_static.argtypes = [vp, i32, i64, vp, i32, i64, vp, i32, i64, i64, i64, vp,
                                        ctypes.POINTER(vp)]
    L.ewg_accumulate_static.restype = i32
    return L


def call_static(L, ids, grad, mg, scratch=None):
    n, H = ids.numel(), mg.shape[1]
    g2 = grad.reshape(n, H)
    code = L.ewg_accumulate_static(
        ids.data_ptr(), _INT64, n, g2.data_ptr(), _BF16 if grad.dtype == torch.bfloat16 else _FP32,
        g2.stride(0), mg.data_ptr(), _BF16 if mg.dtype == torch.bfloat16 else _FP32, mg.shape[0],
        H, mg.stride(0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
        ctypes.byref(scratch) if scratch is not None else None)
    return code


def same_bits(a, b):
    va = a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32)
    vb = b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)
    return bool(torch.equal(va, vb))


@pytest.mark.parametrize("name", ["gpt2_like", "large_vocab"])
def test_static_matches_workspace_entry_point_twice(lib, name):
    """Two calls in a row through each entry point give bitwise the same main_grad."""
    w = workloads.BY_NAME[name]
    ids = torch.from_numpy(workloads.make_ids(w).reshape(-1)).to(DEV)
    grad = workloads.make_grad(w, DEV).reshape(ids.numel(), w.hidden)
    mg_ref = workloads.make_main_grad(w, DEV)
    mg_static = mg_ref.clone()
    ws = ewg.new_workspace(ids.numel(), w.hidden, DEV)
    scratch = ctypes.c_void_p()
    for _ in range(2):
        ewg.accumulate_embedding_wgrad(ids, grad, mg_ref, workspace=ws, check=True)
        assert call_static(lib, ids, grad, mg_static, scratch) == ewg.OK, lib.ewg_last_error()
        status = ctypes.c_int(-1)
        assert lib.ewg_read_status(scratch, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                   ctypes.byref(status)) == ewg.OK
        assert status.value == ewg.OK
        torch.cuda.synchronize()
        assert same_bits(mg_static, mg_ref)


def test_static_call_allocates_nothing(lib):
    """After a first call on the device (which may load the module that holds the array),
    further calls leave the device's free memory exactly as it was."""
    w = workloads.BY_NAME["gpt2_like"]
    ids = torch.from_numpy(workloads.make_ids(w).reshape(-1)).to(DEV)
    grad = workloads.make_grad(w, DEV).reshape(ids.numel(), w.hidden)
    mg = workloads.make_main_grad(w, DEV)
    assert call_static(lib, ids, grad, mg) == ewg.OK, lib.ewg_last_error()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(DEV)[0]
    for _ in range(3):
        assert call_static(lib, ids, grad, mg) == ewg.OK, lib.ewg_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free_before


def test_static_rejects_sizes_beyond_its_scratch(lib):
    w = workloads.scaled(workloads.BY_NAME["long_runs"], num_embeddings=1000)
    n, H = 65536, 7168
    assert ewg.workspace_bytes(n, H) > (64 << 20)
    ids = torch.zeros(n, dtype=torch.int64, device=DEV)
    grad = torch.zeros(n, H, dtype=torch.bfloat16, device=DEV)
    mg = torch.ones(w.num_embeddings, H, dtype=torch.float32, device=DEV)
    assert call_static(lib, ids, grad, mg) == ewg.ERR_UNSUPPORTED
    assert b"static scratch" in lib.ewg_last_error()
    torch.cuda.synchronize()
    assert bool((mg == 1).all())
