"""The bounds-checking build (libewg_debug.so): the same kernels with every index they
derive from the plan checked.  It must give the oracle's bits on ordinary inputs, and
when a plan entry is corrupted from the host it must report EWG_ERR_BOUNDS through the
status word and finish without touching memory outside its buffers.  The corruption is
only ever applied to the checked build."""
import ctypes

import pytest
import torch

import embedding_weight_grad_gb300 as ewg
import workloads
from test_parity_gpu import DEV, assert_same_bits, oracle_expected

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dlib():
    from embedding_weight_grad_gb300 import build
    build.build(debug=True)
    return ewg.debug_lib()


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def status_of(L, ws):
    st = ctypes.c_int(-1)
    assert L.ewg_read_status(ws.data_ptr(), stream(), ctypes.byref(st)) == ewg.OK
    return st.value


def inputs(name, hidden):
    w = workloads.BY_NAME[name]
    if hidden:
        w = workloads.scaled(w, hidden=hidden)
    ids_np = workloads.make_ids(w)
    ids = torch.from_numpy(ids_np.reshape(-1)).to(DEV)
    grad = workloads.make_grad(w, DEV).reshape(ids.numel(), w.hidden)
    mg = workloads.make_main_grad(w, DEV)
    return ids_np, ids, grad, mg


@pytest.mark.parametrize("name,hidden", [("tiny", None), ("long_runs", 264)])
def test_debug_build_matches_oracle(oracle_mod, dlib, name, hidden):
    ids_np, ids, grad, mg = inputs(name, hidden)
    before = mg.clone()
    ws = ewg.new_workspace(ids.numel(), mg.shape[1], DEV)
    a = ewg._Args(ids, grad, mg)
    assert dlib.ewg_accumulate(*a.c_args(), ws.data_ptr(), ws.numel(), stream()) == ewg.OK
    assert status_of(dlib, ws) == ewg.OK
    torch.cuda.synchronize()
    assert_same_bits(mg, oracle_expected(oracle_mod, ids_np, grad, before))


@pytest.mark.parametrize("name,hidden", [("gpt2_like", None), ("long_runs", 264)])
def test_debug_build_reports_a_corrupted_plan(dlib, name, hidden):
    """Descriptor 0 (a chunk of the plan, on either plan path) gets a position beyond the
    last token between ewg_plan and ewg_apply."""
    _, ids, grad, mg = inputs(name, hidden)
    n, H, V = ids.numel(), mg.shape[1], mg.shape[0]
    ws = ewg.new_workspace(n, H, DEV)
    assert dlib.ewg_plan(ids.data_ptr(), 1, n, V, H, ws.data_ptr(), ws.numel(), stream()) == ewg.OK
    assert status_of(dlib, ws) == ewg.OK
    chunks_at = chunk_region_offset(dlib, n, H)
    ws[chunks_at:chunks_at + 4].view(torch.int32).fill_(n + 12345)   # position word 0
    assert dlib.ewg_apply(grad.data_ptr(), ewg._BF16, H, mg.data_ptr(), ewg._FP32 if mg.dtype == torch.float32
                          else ewg._BF16, n, V, H, H, ws.data_ptr(), ws.numel(), stream()) == ewg.OK
    assert status_of(dlib, ws) == ewg.ERR_BOUNDS


def chunk_region_offset(L, n, H):
    """Byte offset of the chunk descriptors in the workspace: after the 256-byte header,
    the partition tables (6 x 128 ints) and four key / position arrays of ceil(n / 2048) *
    2048 words each (internal layout, every region 256-byte aligned)."""
    def up(x):
        return (x + 255) // 256 * 256
    n_pad = -(-n // 2048) * 2048
    off = up(256) + up(6 * 128 * 4)
    return off + 4 * up(n_pad * 4)


def probe(dlib, words, tile, poll_limit):
    out = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    dlib.ewg_debug_lookback_probe.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p]
    assert dlib.ewg_debug_lookback_probe(words.data_ptr(), tile, poll_limit, out.data_ptr(), stream()) == ewg.OK
    torch.cuda.synchronize()
    return out.tolist()


AGG, INC = 1 << 30, 2 << 30   # word formats of the listing's look-back (include/ewg_debug.h)


def test_lookback_sums_its_predecessors(dlib):
    """40 tiles (two batches of 32 predecessors): tile 0 holds an inclusive sum, the others
    their own counts; the probe from tile 39 finds the sum of all 39 and publishes its own."""
    T = 40
    counts = list(range(1, T))                       # tile j has count j + 1
    w = torch.tensor([INC | 1] + [AGG | c for c in counts[1:]] + [0], dtype=torch.int64).to(torch.int32).to(DEV)
    done, excl = probe(dlib, w, T - 1, 1 << 20)
    assert (done, excl) == (1, sum(counts))
    assert int(w[T - 1].item()) & 0xffffffff == (INC | (sum(counts) + 1))


def test_lookback_gives_up_on_a_predecessor_that_never_publishes(dlib):
    """Tile 5's word is never published: the probe must end on its own after its poll limit
    and report that it gave up, without publishing a sum."""
    T = 40
    vals = [INC | 1] + [AGG | (j + 1) for j in range(1, T - 1)] + [0]
    vals[5] = 0
    w = torch.tensor(vals, dtype=torch.int64).to(torch.int32).to(DEV)
    done, _ = probe(dlib, w, T - 1, 2000)
    assert done == 0
    assert int(w[T - 1].item()) == 0


def test_lookback_stops_at_the_closest_inclusive_word(dlib):
    """Tile 20 already holds an inclusive sum: the probe from tile 39 adds tiles 38..21 to
    it and needs nothing older, so an older word that was never published (tile 10) does
    not hold it up."""
    T = 40
    vals = [AGG | (j + 1) for j in range(T - 1)] + [0]
    vals[0] = INC | 1
    vals[20] = INC | 1000
    vals[10] = 0
    w = torch.tensor(vals, dtype=torch.int64).to(torch.int32).to(DEV)
    done, excl = probe(dlib, w, T - 1, 2000)
    assert (done, excl) == (1, 1000 + sum(range(22, 40)))
    assert int(w[T - 1].item()) & 0xffffffff == (INC | (1000 + sum(range(22, 40)) + 1))


@pytest.mark.parametrize("inc_at", [0, 31, 32, 64, 97])
def test_lookback_over_several_batches(dlib, inc_at):
    """100 predecessors, four batches of up to 32, with the closest inclusive word at
    each batch edge and inside a batch: the sum runs from tile 99 back to that word."""
    T = 101
    vals = [AGG | (3 * j + 1) for j in range(T - 1)] + [0]
    vals[inc_at] = INC | 7
    w = torch.tensor(vals, dtype=torch.int64).to(torch.int32).to(DEV)
    done, excl = probe(dlib, w, T - 1, 1 << 20)
    want = 7 + sum(3 * j + 1 for j in range(inc_at + 1, T - 1))
    assert (done, excl) == (1, want)
