"""Calls on several streams at once, and calls captured in a CUDA graph and replayed.

The library keeps no state outside the caller's workspace, so calls on different streams
with different workspaces may overlap on the GPU; every kernel launch is stream-ordered
and allocates nothing, so a call can be captured into a CUDA graph and replayed.  Every
result is compared bit for bit with the oracle applied as many times.
"""
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
from test_parity_gpu import DEV, assert_same_bits, make, oracle_expected

pytestmark = pytest.mark.gpu

# one case on each plan path: hashed (at most 8192 tokens) and multi-tile
CASES = [(6000, 4000, 264), (20000, 5000, 520)]


def test_calls_on_two_streams_overlap_safely(oracle_mod):
    """Three calls each on two streams, enqueued alternately with no synchronisation in
    between (each stream with its own workspace and main_grad)."""
    (n1, V1, H1), (n2, V2, H2) = CASES
    ids1, grad1, mg1 = make(n1, V1, H1, seed=61)
    ids2, grad2, mg2 = make(n2, V2, H2, seed=62)
    before1, before2 = mg1.clone(), mg2.clone()
    i1, i2 = torch.from_numpy(ids1).to(DEV), torch.from_numpy(ids2).to(DEV)
    ws1, ws2 = ewg.new_workspace(n1, H1, DEV), ewg.new_workspace(n2, H2, DEV)
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            ewg.accumulate_embedding_wgrad(i1, grad1, mg1, workspace=ws1)
        with torch.cuda.stream(s2):
            ewg.accumulate_embedding_wgrad(i2, grad2, mg2, workspace=ws2)
    torch.cuda.synchronize()
    assert ewg.read_status(ws1) == ewg.OK and ewg.read_status(ws2) == ewg.OK
    want1, want2 = before1, before2
    for _ in range(3):
        want1 = oracle_expected(oracle_mod, ids1, grad1, want1)
        want2 = oracle_expected(oracle_mod, ids2, grad2, want2)
    assert_same_bits(mg1, want1)
    assert_same_bits(mg2, want2)


@pytest.mark.parametrize("n,V,H", CASES)
def test_captured_call_replays_match_oracle(oracle_mod, n, V, H):
    """One call captured into a CUDA graph (after a first call outside the capture, which
    sets the kernels up), then the graph replayed three times."""
    ids, grad, mg = make(n, V, H, seed=n + 7)
    ids_d = torch.from_numpy(ids).to(DEV)
    ws = ewg.new_workspace(n, H, DEV)
    pristine = mg.clone()
    ewg.accumulate_embedding_wgrad(ids_d, grad, mg, workspace=ws)
    torch.cuda.synchronize()
    mg.copy_(pristine)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ewg.accumulate_embedding_wgrad(ids_d, grad, mg, workspace=ws)
    torch.cuda.synchronize()
    assert_same_bits(mg, pristine)          # capturing runs nothing
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert ewg.read_status(ws) == ewg.OK
    want = pristine
    for _ in range(3):
        want = oracle_expected(oracle_mod, ids, grad, want)
    assert_same_bits(mg, want)
