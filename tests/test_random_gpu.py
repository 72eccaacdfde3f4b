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
