"""The bounded waits of the apply kernel, made to run out from the host.

A fold (the ordered combine of a long run's partial sums) waits on its run's arrival
counter.  Between ewg_plan and ewg_apply the test writes, into the plan's header, an
apply epoch no counter can reach and a short poll limit.  ewg_apply must then end on its
own, ewg_read_status must report EWG_ERR_TIMEOUT, and the same workspace must serve a
fresh plan + apply that matches the oracle bit for bit.  Nothing here faults, traps or
hangs the GPU: every wait in the kernel gives up after a bounded number of polls.
"""
import time

import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from test_parity_gpu import DEV, assert_same_bits, oracle_expected

pytestmark = pytest.mark.gpu

# Byte offsets of two header fields (internal layout; fixed by a static_assert next to
# the header's definition): the apply epoch and the fold poll limit.
EPOCH_AT, SPIN_LIMIT_AT = 40, 44


def poke(ws: torch.Tensor, at: int, value: int):
    ws[at:at + 4].view(torch.int32).fill_(value)


@pytest.mark.parametrize("name,hidden", [("gpt2_like", None), ("long_runs", 512)])
def test_fold_wait_runs_out(oracle_mod, name, hidden):
    w = workloads.BY_NAME[name]
    if hidden:
        w = workloads.scaled(w, hidden=hidden)   # the multi-tile plan at a smaller width
    ids_np = workloads.make_ids(w)
    ids = torch.from_numpy(ids_np.reshape(-1)).to(DEV)
    n, H, V = ids.numel(), w.hidden, w.num_embeddings
    grad = workloads.make_grad(w, DEV).reshape(n, H)
    mg = workloads.make_main_grad(w, DEV)
    pristine = mg.clone()
    ws = ewg.new_workspace(n, H, DEV)

    ewg.plan(ids, V, H, ws)
    poke(ws, EPOCH_AT, 1000)        # targets 1001x what the chunks ever deliver
    poke(ws, SPIN_LIMIT_AT, 4096)   # a few milliseconds of polling per fold
    t0 = time.perf_counter()
    ewg.apply(grad, mg, n, ws)
    status = ewg.read_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == ewg.ERR_TIMEOUT, ewg.lib().ewg_status_string(status)
    assert elapsed < 10.0, f"the kernel took {elapsed:.1f} s to give up"

    # the context and the workspace are still usable: a fresh call is exact
    mg2 = pristine.clone()
    ewg.plan(ids, V, H, ws)
    ewg.apply(grad, mg2, n, ws)
    assert ewg.read_status(ws) == ewg.OK
    torch.cuda.synchronize()
    assert_same_bits(mg2, oracle_expected(oracle_mod, ids_np, grad, pristine))
