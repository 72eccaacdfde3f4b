"""GPU parity of the vocabulary-sharded call: each shard of rows gets, bit for bit, the
rows the whole-table oracle computes, through ewg_accumulate_shard.

Rows of a shard depend only on their own tokens' runs, so splitting the table by rows
and running one call per shard must reproduce the whole-table result exactly; ids of
other shards are skipped, out-of-range ids are still errors.
"""
import numpy as np
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from test_parity_gpu import DEV, assert_same_bits, oracle_expected

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from embedding_weight_grad_gb300 import build
    build.build()
    ewg.lib()


def shards_match_oracle(oracle_mod, ids_np, grad_d, mg_d, bounds, ids_dtype=torch.int64):
    """Runs one sharded call per [bounds[i], bounds[i+1]) on a copy of those rows and
    compares the stitched table with the oracle's whole-table result."""
    expect = oracle_expected(oracle_mod, ids_np, grad_d, mg_d)
    ids_d = torch.from_numpy(ids_np).to(DEV, ids_dtype)
    V = mg_d.shape[0]
    got = torch.empty_like(mg_d)
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        shard = mg_d[b0:b1].clone()
        ewg.accumulate_embedding_wgrad_shard(ids_d, grad_d, shard, b0, V, check=True)
        got[b0:b1] = shard
    torch.cuda.synchronize()
    assert_same_bits(got, expect)


@pytest.mark.parametrize("name", ["gpt2_like", "large_vocab"])
def test_hashed_plan_shards(oracle_mod, name):
    w = workloads.BY_NAME[name]
    V = w.num_embeddings
    # uneven shards; the first holds the hottest ids (Zipf ranks map to small ids)
    shards_match_oracle(oracle_mod, workloads.make_ids(w), workloads.make_grad(w, DEV),
                        workloads.make_main_grad(w, DEV), [0, 3, V // 3, V // 3 + 1, V])


def test_tile_plan_shards(oracle_mod):
    """Above 8192 tokens (multi-tile sort): skipped ids sort after the shard's own keys."""
    w = workloads.scaled(workloads.BY_NAME["large_vocab"], num_tokens=20000,
                         num_embeddings=129280, hidden=520)
    V = w.num_embeddings
    shards_match_oracle(oracle_mod, workloads.make_ids(w), workloads.make_grad(w, DEV),
                        workloads.make_main_grad(w, DEV), [0, 1, 5000, V - 7, V])


def test_long_runs_shards(oracle_mod):
    """The long-runs recipe at a reduced width: a forced run in the last row, heavy folds."""
    w = workloads.scaled(workloads.BY_NAME["long_runs"], hidden=264)
    V = w.num_embeddings
    shards_match_oracle(oracle_mod, workloads.make_ids(w), workloads.make_grad(w, DEV),
                        workloads.make_main_grad(w, DEV), [0, 2, V // 2, V - 1, V])


def test_whole_table_shard_equals_plain_call():
    w = workloads.BY_NAME["gpt2_like"]
    ids = torch.from_numpy(workloads.make_ids(w)).to(DEV)
    grad = workloads.make_grad(w, DEV)
    mg = workloads.make_main_grad(w, DEV)
    a, b = mg.clone(), mg.clone()
    ewg.accumulate_embedding_wgrad(ids, grad, a, check=True)
    ewg.accumulate_embedding_wgrad_shard(ids, grad, b, 0, w.num_embeddings, check=True)
    torch.cuda.synchronize()
    assert_same_bits(b, a)


def test_shard_without_tokens_is_untouched():
    w = workloads.BY_NAME["gpt2_like"]
    ids_np = workloads.make_ids(w)
    V = w.num_embeddings
    absent = np.setdiff1d(np.arange(V - 64, V), ids_np.reshape(-1))
    b0 = int(absent[-1])   # a one-row shard no token falls in
    ids = torch.from_numpy(ids_np).to(DEV)
    grad = workloads.make_grad(w, DEV)
    shard = torch.full((1, w.hidden), float("nan"), device=DEV)
    before = shard.clone()
    ewg.accumulate_embedding_wgrad_shard(ids, grad, shard, b0, V, check=True)
    torch.cuda.synchronize()
    assert torch.equal(shard.view(torch.int32), before.view(torch.int32))


@pytest.mark.parametrize("row_begin,rows", [(-1, 10), (0, 0), (50250, 8), (50257, 1)])
def test_bad_shard_ranges_are_rejected(row_begin, rows):
    w = workloads.BY_NAME["gpt2_like"]
    ids = torch.from_numpy(workloads.make_ids(w)).to(DEV)
    grad = workloads.make_grad(w, DEV)
    shard = torch.zeros((max(rows, 1), w.hidden), device=DEV)
    before = shard.clone()
    if rows == 0:
        shard = shard[:0]
        with pytest.raises((ValueError, ewg.EwgError)):
            ewg.accumulate_embedding_wgrad_shard(ids, grad, shard, row_begin, w.num_embeddings)
        return
    with pytest.raises(ewg.EwgError) as e:
        ewg.accumulate_embedding_wgrad_shard(ids, grad, shard, row_begin, w.num_embeddings)
    assert e.value.code == ewg.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(shard, before)


@pytest.mark.parametrize("n", [5000, 12000])
def test_out_of_range_id_outside_the_shard_is_an_error(n):
    V, H = 40000, 64
    rng = np.random.default_rng(7)
    ids_np = rng.integers(0, V, size=n, dtype=np.int64)
    ids_np[n // 2] = V + 3   # outside the table, and outside the shard
    ids = torch.from_numpy(ids_np).to(DEV)
    grad = torch.randn(n, H, device=DEV)
    shard = torch.zeros((100, H), device=DEV)
    with pytest.raises(ewg.EwgError) as e:
        ewg.accumulate_embedding_wgrad_shard(ids, grad, shard, 200, V, check=True)
    assert e.value.code == ewg.ERR_ID_OUT_OF_RANGE
    assert torch.count_nonzero(shard).item() == 0
