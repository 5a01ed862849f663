"""pkv_kv_indices (paged / CSR block tables of a prepared batch) on the GPU
against the CPU oracle, element by element: kv_indptr, the listed entries and
last_page_len bit-exact; nothing written past the live entries; the capacity
limit and the device checks."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests import oracle_pins
from tests.gpu_helpers import build_states, to_np
from tests.helpers import schedule_arrays

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))
SENTINEL = -7777


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    assert torch.cuda.is_available()
    yield
    torch.cuda.empty_cache()


def _filled(n, value=SENTINEL):
    return torch.full((max(n, 1),), value, dtype=torch.int32, device="cuda")


def _compare(st, orc, batch, ref, wl, extra=64):
    """Every group's paged table from the GPU batch equals the oracle's from
    the oracle batch; entries past the live ones keep the sentinel."""
    n = len(ref["index_mapping"])
    for g, spec in enumerate(wl.groups):
        w_ptr, w_idx, w_last = orc.kv_indices(g, ref["index_mapping"], ref["seq_lens"])
        cap = n * spec.max_blocks_per_req
        out = (_filled(n + 1), _filled(cap + extra), _filled(n))
        st.kv_indices(g, batch.index_mapping, batch.seq_lens, capacity=cap, out=out)
        np.testing.assert_array_equal(to_np(out[0])[:n + 1], w_ptr)
        got = to_np(out[1])
        np.testing.assert_array_equal(got[:w_ptr[n]], w_idx)
        assert (got[w_ptr[n]:] == SENTINEL).all(), "wrote past the live entries"
        np.testing.assert_array_equal(to_np(out[2])[:n], w_last)
    assert st.get_error() == 0


def test_worked_example():
    g = json.load(open(os.path.join(HERE, "golden", "worked_example.json")))
    bs = g["block_size"]
    W = g["fixture_choices"]["max_blocks_per_req"]
    st = pkv.State(16, 64, [(bs, W, 1000)])
    for _ in range(8):
        st.add_request([], 0, [[]])
    st.remove_request(6)
    st.remove_request(7)
    sched = dict(g["schedule_in_output_order"])
    for name in ("A", "B"):
        r = g["requests"][name]
        length = r["completed_tokens"] + sched[name]
        st.add_request([1000 * r["row"] + p for p in range(length)], r["completed_tokens"],
                       [r["blocks"]])
    rows = [g["requests"][nm]["row"] for nm, _ in g["schedule_in_output_order"]]
    ns = [c for _, c in g["schedule_in_output_order"]]
    b = st.prepare_batch(rows, ns)
    indptr, indices, last = st.kv_indices(0, b.index_mapping, b.seq_lens)
    want = g["paged_block_tables"]
    assert to_np(indptr).tolist() == want["kv_indptr"]
    assert to_np(indices)[:want["kv_indptr"][-1]].tolist() == want["kv_indices"]
    assert to_np(last).tolist() == want["last_page_len"]
    assert st.get_error() == 0
    st.close()


CASES = oracle_pins.small_workloads() + [
    workloads.random_small(seed=s, block_sizes=bs, num_requests=nr, max_ctx=mc,
                           max_chunk=ch, window=win)
    for s, bs, nr, mc, ch, win in [
        (30, (16,), 300, 2000, 400, 0),       # several CTAs, ragged tail
        (31, (32, 16), 200, 5000, 900, 0),
        (32, (1,), 50, 60, 30, 0),            # one position per block
        (33, (7, 16, 3), 90, 700, 200, 96),   # sliding window: leading -1 entries
        (34, (16,), 1, 100, 50, 0),           # a single request
        (35, (64,), 513, 3000, 5, 0),         # n not a multiple of 32
        (36, (1, 2, 3, 4, 5, 7, 16, 64), 90, 500, 80, 40),   # PKV_MAX_GROUPS groups
    ]]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"{w.name}-{w.seed}")
def test_parity_small(wl):
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    batch = st.prepare_batch(r, ns)
    ref = orc.prepare_batch(r, ns)
    _compare(st, orc, batch, ref, wl)
    st.close()


FULL = [
    lambda: workloads.tiny(seed=0),
    lambda: workloads.decode_heavy(seed=0),
    lambda: workloads.mixed_prefill(seed=0),
    lambda: workloads.two_groups(seed=0),
    lambda: workloads.large_step(seed=0),
]


@pytest.mark.parametrize("make", FULL, ids=["tiny", "decode_heavy", "mixed_prefill",
                                            "two_groups", "large_step"])
def test_parity_full_size(make):
    """The five configurations at full size, after the device-schedule prepare
    with live tables (the path a graph-captured step takes)."""
    wl = make()
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    d_r = torch.tensor(r, dtype=torch.int32, device="cuda")
    d_n = torch.tensor(ns, dtype=torch.int32, device="cuda")
    batch = st.prepare_batch_device(d_r, d_n, int(ns.sum()), flags=pkv.LIVE_TABLES)
    _compare(st, orc, batch, ref, wl)
    st.close()
    orc.close()


def test_max_batch():
    """n = PKV_MAX_BATCH requests (the largest shared-memory scan), rows in a
    random order, seq_lens from 1 to the full row."""
    rng = np.random.default_rng(9)
    n, bs, W = pkv.MAX_BATCH, 4, 6
    st = pkv.State(n, bs * W, [(bs, W, W * n)])
    orc = oracle.OracleState(n, bs * W, [(bs, W, W * n)])
    perm = rng.permutation(W * n).astype(np.int32)
    for i in range(n):
        k = int(rng.integers(1, W + 1))
        blocks = perm[W * i: W * i + k].tolist()
        toks = rng.integers(0, 1000, bs * k).tolist()
        assert st.add_request(toks, 0, [blocks]) == orc.add_request(toks, 0, [blocks]) == i
    im = rng.permutation(n).astype(np.int32)
    held = np.array([st.row_info(int(r))["num_blocks"][0] for r in im], np.int64)
    sl = np.array([rng.integers(1, h * bs + 1) for h in held], np.int32)
    w_ptr, w_idx, w_last = orc.kv_indices(0, im, sl)
    out = (_filled(n + 1), _filled(n * W + 32), _filled(n))
    st.kv_indices(0, torch.tensor(im, device="cuda"), torch.tensor(sl, device="cuda"),
                  capacity=n * W, out=out)
    np.testing.assert_array_equal(to_np(out[0]), w_ptr)
    got = to_np(out[1])
    np.testing.assert_array_equal(got[:w_ptr[n]], w_idx)
    assert (got[w_ptr[n]:] == SENTINEL).all()
    np.testing.assert_array_equal(to_np(out[2]), w_last)
    assert st.get_error() == 0
    st.close()
    orc.close()


def test_capacity_and_empty():
    wl = workloads.random_small(seed=40, block_sizes=(16,), num_requests=120, max_ctx=3000,
                                max_chunk=300)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    batch = st.prepare_batch(r, ns)
    ref = orc.prepare_batch(r, ns)
    n = len(ns)
    w_ptr, w_idx, w_last = orc.kv_indices(0, ref["index_mapping"], ref["seq_lens"])
    total = int(w_ptr[n])
    # exactly enough room: no error
    out = (_filled(n + 1), _filled(total + 40), _filled(n))
    st.kv_indices(0, batch.index_mapping, batch.seq_lens, capacity=total, out=out)
    np.testing.assert_array_equal(to_np(out[1])[:total], w_idx)
    assert (to_np(out[1])[total:] == SENTINEL).all()
    assert st.get_error() == 0
    # too little: the first `cap` entries, nothing past them, the flag
    cap = total - 37
    out = (_filled(n + 1), _filled(total + 40), _filled(n))
    st.kv_indices(0, batch.index_mapping, batch.seq_lens, capacity=cap, out=out)
    np.testing.assert_array_equal(to_np(out[0]), w_ptr)
    np.testing.assert_array_equal(to_np(out[1])[:cap], w_idx[:cap])
    assert (to_np(out[1])[cap:] == SENTINEL).all()
    np.testing.assert_array_equal(to_np(out[2]), w_last)
    assert st.get_error() == pkv.DEVERR_OUTPUT_FULL
    # n = 0 writes kv_indptr[0] only
    out = (_filled(1), _filled(4), None)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    st.kv_indices(0, empty, empty, capacity=0, out=out)
    assert to_np(out[0]).tolist() == [0]
    assert (to_np(out[1]) == SENTINEL).all()
    assert st.get_error() == 0
    # host checks
    assert st.kv_indices(1, batch.index_mapping, batch.seq_lens, capacity=10,
                         check=False) == pkv.ERR_INVALID_ARG
    assert st.kv_indices(0, batch.index_mapping, batch.seq_lens, capacity=-1,
                         check=False) == pkv.ERR_INVALID_ARG
    st.close()


def test_device_checks():
    """A row outside the table, a zero seq_len and one past W_g pages each get
    0 pages (last_page_len 0) and their bit; the other requests are listed."""
    wl = workloads.random_small(seed=41, block_sizes=(16,), num_requests=10, max_ctx=200,
                                max_chunk=20)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    spec = wl.groups[0]
    im = ref["index_mapping"].copy()
    sl = ref["seq_lens"].copy()
    good = np.ones(len(im), bool)
    im[1] = wl.max_reqs           # outside the table
    sl[3] = 0                     # no positions
    sl[5] = spec.max_blocks_per_req * spec.block_size + 1   # one page too many
    good[[1, 3, 5]] = False
    w_ptr, w_idx, w_last = orc.kv_indices(0, im[good], sl[good])
    n = len(im)
    out = (_filled(n + 1), _filled(n * spec.max_blocks_per_req), _filled(n))
    st.kv_indices(0, torch.tensor(im, device="cuda"), torch.tensor(sl, device="cuda"), out=out)
    ptr = to_np(out[0])
    pages = np.diff(ptr)
    assert pages[~good].tolist() == [0, 0, 0]
    np.testing.assert_array_equal(pages[good], np.diff(w_ptr))
    np.testing.assert_array_equal(to_np(out[1])[:ptr[n]], w_idx)
    last = to_np(out[2])
    assert last[~good].tolist() == [0, 0, 0]
    np.testing.assert_array_equal(last[good], w_last)
    assert st.get_error() == pkv.DEVERR_ROW | pkv.DEVERR_COUNT | pkv.DEVERR_BLOCK
    st.close()
