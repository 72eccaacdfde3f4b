"""GPU parity: the CUDA path against the CPU oracle, bit for bit, through the C ABI.

Every comparison is exact (the method's result is unique bit for bit): touched rows
against the oracle, every other row against a pristine copy.  Inputs follow the
seeded recipe in workloads.py; the oracle sees the same values, copied to the host.
"""
import numpy as np
import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from helpers import bits, golden_case_tensors, golden_expected, load_golden, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from embedding_weight_grad_gb300 import build
    build.build()
    ewg.lib()


def as_bits_t(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def oracle_expected(oracle_mod, ids_np, grad_d, mg_before_d):
    """Expected main_grad (on the device): pristine rows everywhere, oracle rows where an
    id occurs.  The oracle runs on the touched rows only, with ids renumbered densely
    in the same order, which leaves every run and its position order unchanged."""
    flat = ids_np.reshape(-1)
    touched = np.unique(flat)
    dense = np.searchsorted(touched, flat)
    t_idx = torch.from_numpy(touched).to(DEV)
    rows = to_np(mg_before_d.index_select(0, t_idx).cpu()).copy()
    g = to_np(grad_d.reshape(flat.size, -1).cpu())
    oracle_mod.accumulate(dense, g, rows)
    expect = mg_before_d.clone()
    expect.index_copy_(0, t_idx, torch.from_numpy(rows.view(np.int16) if rows.dtype == np.uint16
                                                  else rows).view(mg_before_d.dtype).to(DEV))
    return expect


def assert_same_bits(got: torch.Tensor, want: torch.Tensor):
    eq = as_bits_t(got) == as_bits_t(want)
    if not bool(eq.all()):
        bad = (~eq).nonzero()
        r, c = bad[0].tolist()
        raise AssertionError(f"{int(bad.shape[0])} elements differ; first at row {r} col {c}: "
                             f"got {got[r, c].item()!r} want {want[r, c].item()!r}")


def run_case(oracle_mod, ids_np, grad_d, mg_d, ids_dtype=torch.int64):
    mg_before = mg_d.clone()
    ids_d = torch.from_numpy(ids_np).to(DEV, ids_dtype)
    assert ewg.can_accumulate_embedding_wgrad(ids_d, grad_d, mg_d)
    ewg.accumulate_embedding_wgrad(ids_d, grad_d, mg_d, check=True)
    torch.cuda.synchronize()
    assert_same_bits(mg_d, oracle_expected(oracle_mod, ids_np, grad_d, mg_before))


# --- the five workloads at full size ---------------------------------------------------

@pytest.mark.parametrize("name", [w.name for w in workloads.WORKLOADS])
def test_workload_full_size(oracle_mod, name):
    w = workloads.BY_NAME[name]
    ids = workloads.make_ids(w)
    grad = workloads.make_grad(w, DEV)
    mg = workloads.make_main_grad(w, DEV)
    run_case(oracle_mod, ids, grad, mg)


def test_pytorch_dense_path_matches_oracle(oracle_mod):
    """Black-box pin of the oracle: PyTorch's own CUDA embedding backward (sort-based above
    3072 tokens) followed by main_grad.add_ gives the oracle's values on every touched row.
    The library routine is run, never read."""
    for name in ["gpt2_like", "long_runs"]:
        w = workloads.BY_NAME[name]
        ids = workloads.make_ids(w)
        grad = workloads.make_grad(w, DEV)
        mg = workloads.make_main_grad(w, DEV)
        ids_d = torch.from_numpy(ids).to(DEV)
        dense = torch.ops.aten.embedding_dense_backward(grad.reshape(-1, w.hidden), ids_d.reshape(-1),
                                                        w.num_embeddings, -1, False)
        ref = mg.clone()
        ref.add_(dense)
        expect = oracle_expected(oracle_mod, ids, grad, mg)
        t_idx = torch.from_numpy(np.unique(ids)).to(DEV)
        assert_same_bits(ref.index_select(0, t_idx), expect.index_select(0, t_idx))


# --- hand-derived golden cases, embedded in enough tokens --------------------------------

@pytest.mark.parametrize("case", load_golden("hand_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    ids, grad, mg = golden_case_tensors(case)
    want = golden_expected(case, mg)
    V0, H0 = mg.shape
    reps = 8 // np.gcd(8, H0) if H0 % 8 else 1
    H = H0 * reps                                  # tile columns to a multiple of 8
    n0 = ids.numel()
    pad = ewg.MIN_TOKENS - n0                      # filler tokens, one row each, later ids
    ids_full = torch.cat([ids, torch.arange(V0, V0 + pad)])
    grad_full = torch.cat([grad.repeat(1, reps), torch.ones(pad, H, dtype=grad.dtype)])
    mg_full = torch.cat([mg.repeat(1, reps), torch.zeros(pad, H, dtype=mg.dtype)])
    ids_d, grad_d, mg_d = ids_full.to(DEV), grad_full.to(DEV), mg_full.to(DEV)
    ewg.accumulate_embedding_wgrad(ids_d, grad_d, mg_d, check=True)
    got = mg_d.cpu()
    np.testing.assert_array_equal(bits(to_np(got[:V0])), bits(to_np(want.repeat(1, reps))))
    np.testing.assert_array_equal(bits(to_np(got[V0:])), bits(to_np(torch.ones(pad, H, dtype=mg.dtype))))


# --- shapes, dtypes, layouts and degenerate id patterns ----------------------------------

def make(n, V, H, gdt=torch.bfloat16, mdt=torch.float32, seed=0, ids=None):
    rng = np.random.default_rng(seed)
    if ids is None:
        ids = rng.integers(0, V, size=n, dtype=np.int64)
    grad = workloads.normal((n, H), 1.0, gdt, seed + 1, DEV)
    mg = workloads.normal((V, H), 0.1, mdt, seed + 2, DEV)
    return ids, grad, mg


@pytest.mark.parametrize("n,V,H", [
    (3073, 500, 8),            # fewest tokens, narrowest rows
    (8192, 3000, 264),         # largest single-CTA plan, ragged last column slice
    (8192, 40, 8192),          # hashed plan, 40 long runs over wide rows (four column tiles)
    (4000, 300, 8200),         # hashed plan, rows just past four 2048-column tiles
    (8192, 2, 4096),           # hashed plan, two runs of about 4096 rows each
    (8193, 3000, 1000),        # first multi-CTA plan, ragged tile and slice
    (20000, 129280, 520),      # 17-bit ids, several tiles
    (70001, 1 << 20, 16),      # 20-bit ids (3 radix passes), many tiles
    (5000, 1, 64),             # one token id: a single 5000-row run, no radix pass
    (4100, 2, 128),            # two ids: two long runs
    (12000, 40000, 72),        # mostly single-occurrence runs
    (140000, 100000, 8),       # 69 tiles: several histogram batches per sweep, several
                               # listing look-back rounds
    (300001, 5000, 8),         # 147 tiles, a ragged last one
])
def test_shapes_and_id_patterns(oracle_mod, n, V, H):
    run_case(oracle_mod, *make(n, V, H, seed=n))


def test_four_radix_passes(oracle_mod):
    """Ids of 28 bits (a table of 2^27 + 5 rows): four 7-bit radix passes, the most the
    multi-tile plan makes; the ids are drawn so that both ends of the table occur."""
    V, n, H = (1 << 27) + 5, 20000, 8
    rng = np.random.default_rng(27)
    ids = rng.integers(0, V, size=n, dtype=np.int64)
    ids[:50] = V - 1
    ids[50:120] = 0
    ids[120:140] = 1 << 26
    _, grad, mg = make(n, V, H, torch.bfloat16, torch.bfloat16, seed=27, ids=ids)
    run_case(oracle_mod, ids, grad, mg)


DTYPES = [(torch.bfloat16, torch.float32), (torch.bfloat16, torch.bfloat16),
          (torch.float32, torch.float32), (torch.float32, torch.bfloat16)]


@pytest.mark.parametrize("gdt,mdt", DTYPES)
def test_dtype_matrix(oracle_mod, gdt, mdt):
    ids = workloads.zipf_ids(np.random.default_rng(3), 20000, 1.2, 12000)
    run_case(oracle_mod, *make(12000, 20000, 392, gdt, mdt, seed=5, ids=ids))


@pytest.mark.parametrize("gdt,mdt", DTYPES)
def test_dtype_matrix_hashed_plan(oracle_mod, gdt, mdt):
    """The four dtype pairs at 8000 tokens (the hashed plan): Zipf ids, so long runs with
    their folds and single-chunk runs both occur."""
    ids = workloads.zipf_ids(np.random.default_rng(13), 20000, 1.2, 8000)
    run_case(oracle_mod, *make(8000, 20000, 392, gdt, mdt, seed=15, ids=ids))


def test_int32_ids_and_strided_tensors(oracle_mod):
    n, V, H = 9000, 7000, 256
    ids = workloads.zipf_ids(np.random.default_rng(4), V, 1.1, n)
    wide_g = workloads.normal((n, H + 64), 1.0, torch.bfloat16, 7, DEV)
    wide_m = workloads.normal((V, H + 32), 0.1, torch.float32, 8, DEV)
    grad = wide_g[:, 32:32 + H]          # row stride H + 64, 64-byte offset
    mg = wide_m[:, :H]                   # row stride H + 32
    mg_before = wide_m.clone()
    ids_d = torch.from_numpy(ids).to(DEV, torch.int32)
    ewg.accumulate_embedding_wgrad(ids_d, grad, mg, check=True)
    expect = oracle_expected(oracle_mod, ids, grad.contiguous(), mg_before[:, :H].contiguous())
    assert_same_bits(wide_m[:, :H].contiguous(), expect)
    assert_same_bits(wide_m[:, H:].contiguous(), mg_before[:, H:].contiguous())


def test_runs_at_chunk_boundaries(oracle_mod):
    """Runs of exactly 1, 9, 10, 11, 19, 20, 21 and 101 rows, interleaved in position."""
    lengths = [1, 9, 10, 11, 19, 20, 21, 101] * 40
    ids = np.repeat(np.arange(len(lengths)), lengths)
    ids = np.random.default_rng(9).permutation(ids)
    run_case(oracle_mod, *make(ids.size, len(lengths), 136, seed=9, ids=ids))


def test_runs_at_chunk_boundaries_hashed_plan(oracle_mod):
    """The same run lengths plus 30, 31, 40 and 41 rows in 8000 tokens (the hashed plan),
    the other positions single-row runs of their own ids."""
    lengths = [1, 9, 10, 11, 19, 20, 21, 30, 31, 40, 41, 101] * 20
    ids = np.repeat(np.arange(len(lengths)), lengths)
    ids = np.random.default_rng(19).permutation(ids)
    ids = np.concatenate([ids, np.arange(1000, 1000 + 8000 - ids.size)])
    run_case(oracle_mod, *make(ids.size, 9000, 200, seed=19, ids=ids))


def test_repeated_calls_accumulate(oracle_mod):
    ids, grad, mg = make(10000, 3000, 256, seed=21)
    mg_before = mg.clone()
    ids_d = torch.from_numpy(ids).to(DEV)
    ws = ewg.new_workspace(ids.size, 256, DEV)
    for _ in range(2):
        ewg.accumulate_embedding_wgrad(ids_d, grad, mg, workspace=ws, check=True)
    once = oracle_expected(oracle_mod, ids, grad, mg_before)
    twice = oracle_expected(oracle_mod, ids, grad, once)
    assert_same_bits(mg, twice)


def test_plan_then_apply_matches_accumulate(oracle_mod):
    n, V, H = 9000, 5000, 512
    ids, grad, mg = make(n, V, H, seed=31)
    mg2 = mg.clone()
    ids_d = torch.from_numpy(ids).to(DEV)
    ws = ewg.new_workspace(n, H, DEV)
    ewg.plan(ids_d, V, H, ws)
    ewg.apply(grad, mg, n, ws)
    assert ewg.read_status(ws) == ewg.OK
    ewg.accumulate_embedding_wgrad(ids_d, grad, mg2, check=True)
    assert_same_bits(mg, mg2)


def test_apply_with_a_mismatched_plan_writes_nothing():
    n, V, H = 9000, 5000, 512
    ids, grad, mg = make(n, V, H, seed=32)
    before = mg.clone()
    ws = ewg.new_workspace(n, H, DEV)
    ewg.plan(torch.from_numpy(ids).to(DEV), V, H, ws)
    ewg.apply(grad, mg[: V - 1], n, ws)              # num_embeddings differs from the plan
    assert ewg.read_status(ws) == ewg.ERR_INVALID
    assert_same_bits(mg, before)


def test_out_of_range_ids_leave_main_grad_untouched():
    for bad in (-1, 5000, 1 << 40):
        ids, grad, mg = make(9000, 5000, 256, seed=41)
        ids[1234] = bad
        before = mg.clone()
        with pytest.raises(ewg.EwgError) as e:
            ewg.accumulate_embedding_wgrad(torch.from_numpy(ids).to(DEV), grad, mg, check=True)
        assert e.value.code == ewg.ERR_ID_OUT_OF_RANGE
        assert_same_bits(mg, before)
    ids, grad, mg = make(4000, 5000, 256, seed=42)     # single-CTA plan path
    ids[17] = 5000
    before = mg.clone()
    with pytest.raises(ewg.EwgError):
        ewg.accumulate_embedding_wgrad(torch.from_numpy(ids).to(DEV), grad, mg, check=True)
    assert_same_bits(mg, before)


def test_unsupported_inputs_are_rejected_before_any_work():
    ids, grad, mg = make(4000, 1000, 256, seed=51)
    ids_d = torch.from_numpy(ids).to(DEV)
    before = mg.clone()
    cases = [
        (ids_d[:3072], grad[:3072], mg),                       # too few tokens
        (ids_d, grad[:, :252], mg[:, :252]),                   # hidden not a multiple of 8
        (ids_d, grad.half(), mg),                              # fp16 grad
        (ids_d.cpu(), grad, mg),                               # ids on the host
        (ids_d, grad, mg.t().contiguous().t()),                # column-major main_grad
        (ids_d.float(), grad, mg),                             # float ids
    ]
    for i, g, m in cases:
        assert not ewg.can_accumulate_embedding_wgrad(i, g, m)
        with pytest.raises(ValueError):
            ewg.accumulate_embedding_wgrad(i, g, m)
    assert_same_bits(mg, before)
    # misaligned: a grad view starting 2 bytes into a row
    wide = torch.zeros(4000, 264, dtype=torch.bfloat16, device=DEV)
    assert not ewg.can_accumulate_embedding_wgrad(ids_d, wide[:, 1:257], mg)


def test_tensors_overlapping_the_workspace_are_rejected():
    """One allocation carved into the workspace and main_grad (or grad) so that they share
    bytes: every entry point that writes the workspace must refuse before any work."""
    ids, grad, mg = make(4000, 1000, 256, seed=52)
    ids_d = torch.from_numpy(ids).to(DEV)
    need = ewg.workspace_bytes(4000, 256)
    L = ewg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    buf = torch.zeros(need + max(mg.numel() * 4, grad.numel() * 2), dtype=torch.uint8, device=DEV)
    ws = buf[:need]
    # main_grad starts inside the workspace (256-byte aligned, half way in)
    mg_in = buf[need // 512 * 256:].view(torch.float32)[: mg.numel()].view(mg.shape)
    mg_in.copy_(mg)
    before = mg_in.clone()
    a = ewg._Args(ids_d, grad, mg_in)
    code = L.ewg_accumulate(*a.c_args(), ws.data_ptr(), need, stream)
    assert code == ewg.ERR_UNSUPPORTED and b"overlaps the workspace" in L.ewg_last_error()
    code = L.ewg_apply(grad.data_ptr(), ewg._BF16, 256, mg_in.data_ptr(), ewg._FP32, 4000, 1000,
                       256, 256, ws.data_ptr(), need, stream)
    assert code == ewg.ERR_UNSUPPORTED and b"overlaps the workspace" in L.ewg_last_error()
    # grad inside the workspace
    g_in = buf[need // 512 * 256:].view(torch.bfloat16)[: grad.numel()].view(grad.shape)
    b = ewg._Args(ids_d, g_in, mg)
    code = L.ewg_accumulate(*b.c_args(), ws.data_ptr(), need, stream)
    assert code == ewg.ERR_UNSUPPORTED and b"overlaps the workspace" in L.ewg_last_error()
    torch.cuda.synchronize()
    assert_same_bits(mg_in, before)


def test_deterministic_across_runs(oracle_mod):
    w = workloads.scaled(workloads.BY_NAME["long_runs"], hidden=512)
    ids = workloads.make_ids(w)
    grad = workloads.make_grad(w, DEV)
    mg0 = workloads.make_main_grad(w, DEV)
    outs = []
    for _ in range(3):
        mg = mg0.clone()
        ewg.accumulate_embedding_wgrad(torch.from_numpy(ids).to(DEV), grad, mg, check=True)
        outs.append(mg)
    assert_same_bits(outs[0], outs[1])
    assert_same_bits(outs[0], outs[2])
    assert_same_bits(outs[0], oracle_expected(oracle_mod, ids, grad, mg0))
