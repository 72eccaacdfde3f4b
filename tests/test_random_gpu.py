"""GPU parity over seeded random configurations: token counts on both plan paths, table
sizes, hidden sizes (ragged against every tile and slice width), both dtypes of grad and
main_grad, int32 and int64 ids, and id mixes from uniform to one dominant run.  Every
case is compared with the oracle bit for bit, like the fixed cases."""
import numpy as np
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from test_parity_gpu import DEV, make, run_case

pytestmark = pytest.mark.gpu

DTYPES = (torch.bfloat16, torch.float32)


def random_case(seed: int):
    rng = np.random.default_rng(10_000 + seed)
    band = int(rng.integers(0, 3))                  # narrow, medium and wide rows
    H = 8 * int(rng.integers(*[(1, 33), (33, 326), (326, 1101)][band]))
    n = int(rng.integers(ewg.MIN_TOKENS, max(ewg.MIN_TOKENS + 1, min(60_000, 60_000_000 // H))))
    tables = [V for V in (1, 7, 100, 5_000, 129_280, 1 << 20) if V * H * 4 <= (4 << 30)]
    V = int(rng.choice(tables))
    kind = rng.choice(["uniform", "zipf", "forced"])
    if kind == "uniform" or V < 8:
        ids = rng.integers(0, V, size=n, dtype=np.int64)
    else:
        ids = workloads.zipf_ids(rng, V, float(rng.uniform(0.8, 1.6)), n)
        if kind == "forced":   # one id, anywhere in the table, at a random share of positions
            where = rng.choice(n, size=int(n * rng.uniform(0.05, 0.6)), replace=False)
            ids[where] = int(rng.integers(0, V))
    gdt, mdt = DTYPES[int(rng.integers(0, 2))], DTYPES[int(rng.integers(0, 2))]
    ids_dtype = torch.int32 if rng.integers(0, 2) else torch.int64
    return ids, n, V, H, gdt, mdt, ids_dtype


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(oracle_mod, seed):
    ids, n, V, H, gdt, mdt, ids_dtype = random_case(seed)
    _, grad, mg = make(n, V, H, gdt, mdt, seed=seed, ids=ids)
    run_case(oracle_mod, ids, grad, mg, ids_dtype=ids_dtype)


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().contiguous().pin_memory()


@pytest.mark.parametrize("seed", range(24, 42))
def test_random_configuration_other_entry_points(oracle_mod, seed):
    """The same random configurations through the other entry points, in turn: one plan
    applied twice (ewg_plan, then ewg_apply twice: the apply's epoch lets a plan serve
    repeated calls), a random row range of the table (ewg_accumulate_shard), and ids and
    grad in pinned host memory (ewg_accumulate_host)."""
    from test_parity_gpu import assert_same_bits, oracle_expected
    ids, n, V, H, gdt, mdt, ids_dtype = random_case(seed)
    _, grad, mg = make(n, V, H, gdt, mdt, seed=seed, ids=ids)
    ids_d = torch.from_numpy(ids).to(DEV, ids_dtype)
    before = mg.clone()
    entry = ["plan_twice", "shard", "host"][seed % 3]
    if entry == "plan_twice":
        ws = ewg.new_workspace(n, H, DEV)
        ewg.plan(ids_d, V, H, ws)
        ewg.apply(grad, mg, n, ws)
        ewg.apply(grad, mg, n, ws)
        assert ewg.read_status(ws) == ewg.OK
        want = oracle_expected(oracle_mod, ids, grad, oracle_expected(oracle_mod, ids, grad, before))
        assert_same_bits(mg, want)
    elif entry == "shard":
        rng = np.random.default_rng(20_000 + seed)
        b0 = int(rng.integers(0, V))
        b1 = int(rng.integers(b0 + 1, V + 1))
        shard = mg[b0:b1].clone()
        ewg.accumulate_embedding_wgrad_shard(ids_d, grad, shard, b0, V, check=True)
        want = oracle_expected(oracle_mod, ids, grad, before)
        assert_same_bits(shard, want[b0:b1])
    else:
        ewg.accumulate_embedding_wgrad_from_host(_pinned(ids_d), _pinned(grad), mg, check=True)
        assert_same_bits(mg, oracle_expected(oracle_mod, ids, grad, before))
