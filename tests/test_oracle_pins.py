"""Pins for the CPU oracle: facts fixed by the pages and by arithmetic, not by the oracle.

Source of the method: Megatron Core API docs, core.fusions.fused_embedding_wgrad,
module docstring (sort-based order of PyTorch's embedding backward, one rounding to
the gradient dtype, fp32 add into main_grad, absent rows untouched).

Each test is chosen so that a plausible slip in the oracle fails it: a dropped or
duplicated row, a wrong position or id mapping, a sign error, chunks not aligned to
the run start, a chunk length other than 10, an extra or missing rounding, the add
done in the wrong precision, absent rows written.
"""
import numpy as np
import pytest
import torch

import workloads
from helpers import bits, from_np, golden_case_tensors, golden_expected, load_golden, to_np


def run_oracle(oracle_mod, ids, grad, mg, **kw):
    out = to_np(mg).copy()
    oracle_mod.accumulate(ids.numpy() if torch.is_tensor(ids) else ids, to_np(grad), out, **kw)
    return out


# --- hand-derived golden cases ------------------------------------------------------

@pytest.mark.parametrize("case", load_golden("hand_cases.json")["cases"], ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    ids, grad, mg = golden_case_tensors(case)
    out = run_oracle(oracle_mod, ids, grad, mg)
    want = to_np(golden_expected(case, mg))
    np.testing.assert_array_equal(bits(out), bits(want))


# --- P1: a token that occurs once ---------------------------------------------------

@pytest.mark.parametrize("gdt,mdt", [(torch.bfloat16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                     (torch.float32, torch.float32), (torch.float32, torch.bfloat16)])
def test_single_occurrence_closed_form(oracle_mod, gdt, mdt):
    """One occurrence: the weight-gradient row is the grad row itself (0 + 0 + g = g, and
    rounding a value already in grad's dtype is exact), so the result is round_mg(mg + g)."""
    rng = np.random.default_rng(11)
    V, H, n = 9000, 40, 4000
    ids = rng.permutation(V)[:n].astype(np.int64)
    grad = workloads.normal((n, H), 1.0, gdt, 5)
    mg = workloads.normal((V, H), 0.5, mdt, 6)
    out = run_oracle(oracle_mod, ids, grad, mg)
    want = mg.clone()
    want[torch.from_numpy(ids)] = (mg[torch.from_numpy(ids)].float() + grad.float()).to(mdt)
    np.testing.assert_array_equal(bits(out), bits(to_np(want)))


# --- P2: integer gradients make every fp32 sum exact --------------------------------

@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float32])
def test_integer_grads_order_independent(oracle_mod, gdt):
    """Integer grads in [-4, 4]: every partial and total is an integer below 2^24, so fp32
    arithmetic is exact in any order and w = round_g(exact integer sum)."""
    rng = np.random.default_rng(12)
    V, H, n = 300, 24, 20000
    ids = workloads.zipf_ids(rng, V, 1.2, n)
    g_int = rng.integers(-4, 5, size=(n, H))
    grad = torch.from_numpy(g_int.astype(np.float32)).to(gdt)
    mg_int = rng.integers(-1000, 1000, size=(V, H))
    mg = torch.from_numpy(mg_int.astype(np.float32))
    out = run_oracle(oracle_mod, ids, grad, mg)

    exact = np.zeros((V, H), dtype=np.int64)
    np.add.at(exact, ids, g_int)
    w = torch.from_numpy(exact.astype(np.float32)).to(gdt).float()   # the one rounding
    want = mg.clone()
    present = np.unique(ids)
    want[present] = mg[present] + w[present]
    np.testing.assert_array_equal(bits(out), bits(to_np(want)))
    assert np.abs(exact).max() > 256  # some bf16 roundings really happen


# --- P3: within one rounding of the exact (fp64) dense result ----------------------

@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float32])
def test_fp64_dense_bound(oracle_mod, gdt):
    """|w - S| <= u_g |S| + 2 (L + 1) 2^-24 sum|g|, S the fp64 zero-fill + index_add row,
    u_g = 2^-8 for bf16 and 0 for fp32, L the run length (recursive-summation bound)."""
    rng = np.random.default_rng(13)
    V, H, n = 2000, 64, 30000
    ids = workloads.zipf_ids(rng, V, 1.1, n)
    grad = workloads.normal((n, H), 1.0, gdt, 7)
    uniq, w = oracle_mod.weight_grad(ids, to_np(grad), V)

    g64 = grad.double().numpy()
    dense = np.zeros((V, H))
    np.add.at(dense, ids, g64)
    absum = np.zeros((V, H))
    np.add.at(absum, ids, np.abs(g64))
    L = np.bincount(ids, minlength=V)
    np.testing.assert_array_equal(uniq, np.nonzero(L)[0])
    S = dense[uniq]
    u = 2.0 ** -8 if gdt == torch.bfloat16 else 0.0
    bound = u * np.abs(S) + 2 * (L[uniq, None] + 1) * 2.0 ** -24 * absum[uniq]
    err = np.abs(w.astype(np.float64) - S)
    assert (err <= bound).all(), float((err - bound).max())
    assert L.max() > 100


# --- P4: absent rows are bitwise untouched ------------------------------------------

@pytest.mark.parametrize("mdt", [torch.float32, torch.bfloat16])
def test_absent_rows_untouched(oracle_mod, mdt):
    """Rows of ids that do not occur keep every bit, including -0.0, NaN payloads and
    infinities (adding 0 as the dense path does would change -0.0 to +0.0)."""
    rng = np.random.default_rng(14)
    V, H, n = 512, 16, 3500
    ids = rng.integers(0, V // 2, size=n) * 2   # odd rows never occur
    grad = workloads.normal((n, H), 1.0, torch.bfloat16, 8)
    mg = workloads.normal((V, H), 1.0, mdt, 9)
    raw = to_np(mg).copy()
    if mdt == torch.float32:
        specials = np.array([0x80000000, 0x7fc01234, 0xff800000, 0x00000001, 0x7f800000],
                            dtype=np.uint32).view(np.float32)
    else:
        specials = np.array([0x8000, 0x7fc1, 0xff80, 0x0001, 0x7f80], dtype=np.uint16)
    odd = np.arange(1, V, 2)
    raw[np.ix_(odd, np.arange(len(specials)))] = specials
    before = raw.copy()
    oracle_mod.accumulate(ids, to_np(grad), raw)
    np.testing.assert_array_equal(bits(raw[odd]), bits(before[odd]))
    assert not np.array_equal(bits(raw[::2]), bits(before[::2]))


# --- runs of at most 10 rows: one partial sum, i.e. the sequential sum ---------------

def test_short_runs_are_sequential_sums(oracle_mod):
    """A run of L <= 10 rows is a single chunk, so w = round_g(g_0 + g_1 + ... ) summed in
    position order; numpy's float32 cumulative sum is that sequential sum."""
    rng = np.random.default_rng(15)
    V, H = 4000, 32
    counts = rng.integers(1, 11, size=V)
    ids = rng.permutation(np.repeat(np.arange(V), counts))
    n = ids.size
    grad = workloads.normal((n, H), 1.0, torch.bfloat16, 10)
    uniq, w = oracle_mod.weight_grad(ids, to_np(grad), V)
    g32 = grad.float().numpy()
    for t in rng.choice(V, size=200, replace=False):
        rows = g32[np.nonzero(ids == t)[0]]          # position order
        seq = np.cumsum(rows, axis=0, dtype=np.float32)[-1]
        want = torch.from_numpy(seq).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(bits(w[np.searchsorted(uniq, t)]), bits(want))


# --- chunking is aligned to each run, not to global slots or ids ---------------------

def test_relabel_invariance(oracle_mod):
    """Each run's row depends only on its own rows in position order.  Relabelling the
    ids by a random bijection moves runs to other sorted slots; every row must follow its
    token unchanged (chunks aligned to global slots, or rows from a neighbouring run,
    would change values)."""
    rng = np.random.default_rng(16)
    V, H, n = 700, 16, 12000
    ids = workloads.zipf_ids(rng, V, 1.05, n)
    grad = workloads.normal((n, H), 1.0, torch.bfloat16, 11)
    perm = rng.permutation(V)
    u1, w1 = oracle_mod.weight_grad(ids, to_np(grad), V)
    u2, w2 = oracle_mod.weight_grad(perm[ids], to_np(grad), V)
    order = np.searchsorted(u2, perm[u1])
    np.testing.assert_array_equal(bits(w1), bits(w2[order]))


# --- step 1 on its own -----------------------------------------------------------------

def test_sort_pairs_matches_stable_argsort(oracle_mod):
    rng = np.random.default_rng(17)
    ids = workloads.zipf_ids(rng, 5000, 1.1, 9000)
    sid, spos = oracle_mod.sort_pairs(ids, 5000)
    ref = np.argsort(ids, kind="stable")
    np.testing.assert_array_equal(spos, ref)
    np.testing.assert_array_equal(sid, ids[ref])


# --- the rounding routine against a library conversion ---------------------------------

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(18)
    with np.errstate(over="ignore"):
        x = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 128, 200000))).astype(np.float32)
    u = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    ties = ((rng.integers(0, 2**16, 5000).astype(np.uint32) << 16) | 0x8000).astype(np.uint32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.finfo(np.float32).max,
                        -np.finfo(np.float32).max, 1e-45, -1e-45, 1.0 + 2**-8, 1.0 + 3 * 2**-8],
                       dtype=np.float32)
    allx = np.concatenate([x, u.view(np.float32), ties.view(np.float32), special])
    allx = allx[~np.isnan(allx)]
    got = oracle_mod.round_to_bf16(allx)
    want = to_np(torch.from_numpy(allx).to(torch.bfloat16))
    np.testing.assert_array_equal(got, want)
    nan = oracle_mod.round_to_bf16(np.array([np.nan, -np.nan], dtype=np.float32))
    assert np.isnan(oracle_mod.bf16_bits_to_float(nan)).all()


# --- invariants of the implementation around the arithmetic -----------------------------

def test_threads_stride_dtype_and_shape_invariance(oracle_mod):
    """Thread count, an int32 copy of the ids, a strided grad view and a 2-D ids shape must
    give bitwise the same main_grad."""
    w = workloads.scaled(workloads.BY_NAME["gpt2_like"], num_embeddings=3000, hidden=48)
    ids = workloads.make_ids(w)                       # [4, 2048]
    grad = workloads.make_grad(w)                     # [4, 2048, 48] bf16
    mg = workloads.make_main_grad(w)
    ref = run_oracle(oracle_mod, ids, grad, mg, num_threads=1)
    assert np.array_equal(bits(run_oracle(oracle_mod, ids, grad, mg, num_threads=8)), bits(ref))
    assert np.array_equal(bits(run_oracle(oracle_mod, ids.astype(np.int32), grad, mg)), bits(ref))
    wide = torch.zeros(ids.size, 80, dtype=torch.bfloat16)
    wide[:, 16:64] = grad.reshape(-1, 48)
    strided = to_np(wide)[:, 16:64]
    out = to_np(mg).copy()
    oracle_mod.accumulate(ids.reshape(-1), strided, out)
    assert np.array_equal(bits(out), bits(ref))


def test_out_of_range_id_is_an_error(oracle_mod):
    ids = np.array([0, 1, 5, 2], dtype=np.int64)
    grad = np.zeros((4, 8), dtype=np.float32)
    mg = np.ones((5, 8), dtype=np.float32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.accumulate(ids, grad, mg)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.accumulate(np.array([0, -1, 1, 2]), grad, mg)
    assert (mg == 1).all()


def test_workload_recipe_shapes():
    """The seeded recipe gives the stated shapes, ranges and the forced long run."""
    for w in workloads.WORKLOADS[:4]:
        ids = workloads.make_ids(w)
        assert ids.shape == w.ids_shape and ids.dtype == np.int64
        assert ids.min() >= 0 and ids.max() < w.num_embeddings
    lr = workloads.BY_NAME["long_runs"]
    ids = workloads.make_ids(lr).reshape(-1)
    assert (ids == lr.num_embeddings - 1).sum() >= round(0.2 * ids.size)
    assert np.array_equal(workloads.make_ids(lr).reshape(-1), ids)   # seeded


def test_zipf_recipe_frequencies():
    """The Zipf ids follow P(id = k - 1) proportional to k**-s: the counts of the first
    ranks lie within 5 standard deviations of n P, computed here from the closed-form
    normaliser (a partial zeta sum), and hot ids are the small ones."""
    rng = np.random.default_rng(7)
    V, s, n = 129280, 1.1, 200000
    ids = workloads.zipf_ids(rng, V, s, n)
    norm = float(np.sum(np.arange(1, V + 1, dtype=np.float64) ** -s))
    counts = np.bincount(ids, minlength=V)
    for k in range(1, 6):
        p = k ** -s / norm
        mean, sd = n * p, (n * p * (1 - p)) ** 0.5
        assert abs(counts[k - 1] - mean) < 5 * sd, (k, counts[k - 1], mean)
    assert counts[0] > counts[1] > counts[2] > counts[10]
    assert ids.min() >= 0 and ids.max() < V
