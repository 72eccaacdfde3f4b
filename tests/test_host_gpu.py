"""The host-input entry point (ewg_accumulate_host): ids and grad start in pinned host
memory and the library copies them in.  main_grad must end up with the oracle's bits,
the same as when the same inputs are passed from device memory; the wrapper must keep
the pinned inputs alive until the stream has passed the call."""
import ctypes

import numpy as np
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from test_parity_gpu import DEV, assert_same_bits, oracle_expected

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,ids_dtype", [("gpt2_like", torch.int64), ("large_vocab", torch.int32),
                                            ("long_runs", torch.int64)])
def test_host_inputs_match_device_inputs(name, ids_dtype):
    w = workloads.BY_NAME[name]
    if name == "long_runs":        # the multi-tile plan at a smaller hidden size
        w = workloads.scaled(w, hidden=512)
    ids = torch.from_numpy(workloads.make_ids(w).reshape(-1)).to(ids_dtype)
    grad_d = workloads.make_grad(w, DEV).reshape(ids.numel(), w.hidden)
    mg_dev = workloads.make_main_grad(w, DEV)
    mg_host_path = mg_dev.clone()
    ids_pin, grad_pin = ids.pin_memory(), grad_d.cpu().pin_memory()
    ws = ewg.new_host_workspace(ids.numel(), w.hidden, ids.dtype, grad_pin.dtype, DEV)
    for _ in range(2):             # the second call reuses the workspace and the copy stream
        ewg.accumulate_embedding_wgrad(ids.to(DEV), grad_d, mg_dev, check=True)
        ewg.accumulate_embedding_wgrad_from_host(ids_pin, grad_pin, mg_host_path, workspace=ws,
                                                 check=True)
        torch.cuda.synchronize()
        assert_same_bits(mg_host_path, mg_dev)


def test_host_inputs_must_be_pinned():
    n, H, V = 4096, 64, 1000
    ids = np.zeros(n, dtype=np.int64)
    grad = np.zeros((n, H), dtype=np.float32)
    mg = torch.ones(V, H, device=DEV)
    ws = ewg.new_host_workspace(n, H, torch.int64, torch.float32, DEV)
    L = ewg.lib()
    code = L.ewg_accumulate_host(ids.ctypes.data, ewg._ID_CODES[torch.int64], n, grad.ctypes.data,
                                 ewg._FLOAT_CODES[torch.float32], mg.data_ptr(),
                                 ewg._FLOAT_CODES[torch.float32], V, H, H, ws.data_ptr(), ws.numel(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == ewg.ERR_UNSUPPORTED and b"page-locked" in L.ewg_last_error()
    with pytest.raises(ValueError):
        ewg.accumulate_embedding_wgrad_from_host(torch.zeros(n, dtype=torch.int64),
                                                 torch.zeros(n, H), mg)
    torch.cuda.synchronize()
    assert bool((mg == 1).all())


@pytest.mark.parametrize("name,ids_dtype", [("large_vocab", torch.int64), ("tiny", torch.int32)])
def test_host_inputs_match_oracle(oracle_mod, name, ids_dtype):
    """The call the bench's end-to-end figure times, compared with the oracle directly."""
    w = workloads.BY_NAME[name]
    ids_np = workloads.make_ids(w)
    ids_pin = torch.from_numpy(ids_np.reshape(-1)).to(ids_dtype).pin_memory()
    grad_pin = workloads.make_grad(w).reshape(ids_pin.numel(), w.hidden).pin_memory()
    mg = workloads.make_main_grad(w, DEV)
    before = mg.clone()
    ewg.accumulate_embedding_wgrad_from_host(ids_pin, grad_pin, mg, check=True)
    torch.cuda.synchronize()
    assert_same_bits(mg, oracle_expected(oracle_mod, ids_np, grad_pin.to(DEV), before))


def test_dropped_pinned_inputs_stay_valid_until_the_copy_has_run():
    """Temporaries pinned for the call and dropped at once: while the stream is still busy
    with earlier work (so the copies have not run), new pinned buffers of the same size
    are allocated and overwritten.  The copies must still read the original values."""
    w = workloads.scaled(workloads.BY_NAME["gpt2_like"], hidden=512)
    ids = torch.from_numpy(workloads.make_ids(w).reshape(-1))
    grad = workloads.make_grad(w).reshape(ids.numel(), w.hidden)
    mg_ref = workloads.make_main_grad(w, DEV)
    mg = mg_ref.clone()
    ewg.accumulate_embedding_wgrad(ids.to(DEV), grad.to(DEV), mg_ref, check=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)       # keeps the stream busy for a while (device cycles)
    ewg.accumulate_embedding_wgrad_from_host(ids.pin_memory(), grad.pin_memory(), mg)
    junk_ids = torch.empty_like(ids).pin_memory()
    junk_grad = torch.empty_like(grad).pin_memory()
    junk_ids.fill_(7)
    junk_grad.fill_(1e30)
    torch.cuda.synchronize()
    assert_same_bits(mg, mg_ref)
    del junk_ids, junk_grad
