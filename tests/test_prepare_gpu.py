"""prepare_batch on the GPU against the CPU oracle, element by element.

Every output (index_mapping, query_start_loc, seq_lens, positions, input_ids,
and per KV-cache group the gathered block tables and slot_mapping) must be
bit-exact; the request-state table must match the oracle's row for row."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests import oracle_pins
from tests.gpu_helpers import build_states, compare_batch, prepare_both, to_np
from tests.helpers import schedule_arrays

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    assert torch.cuda.is_available()
    yield
    torch.cuda.empty_cache()


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
    for name, want_row in (("A", 6), ("B", 7)):
        r = g["requests"][name]
        length = r["completed_tokens"] + sched[name]
        toks = [1000 * r["row"] + p for p in range(length)]
        assert st.add_request(toks, r["completed_tokens"], [r["blocks"]]) == want_row
    rows = [g["requests"][nm]["row"] for nm, _ in g["schedule_in_output_order"]]
    ns = [c for _, c in g["schedule_in_output_order"]]
    b = st.prepare_batch(rows, ns)
    pr = g["printed_on_the_pages"]
    assert to_np(b.query_start_loc).tolist() == pr["query_start_loc"]
    assert to_np(b.positions).tolist() == pr["positions"]
    assert int(to_np(b.slot_mapping[0])[0]) == pr["first_token_of_B"]["slot"]
    der = g["derived_from_the_definitions"]
    assert to_np(b.index_mapping).tolist() == der["index_mapping"]
    assert to_np(b.seq_lens).tolist() == der["seq_lens"]
    assert to_np(b.slot_mapping[0]).tolist() == der["slot_mapping"]
    fx = g["fixture_choices"]
    assert to_np(b.input_ids).tolist() == fx["input_ids"]
    assert to_np(b.block_tables[0]).tolist() == fx["input_block_tables"]
    assert st.get_error() == 0
    st.close()


SMALL = oracle_pins.small_workloads() + [
    workloads.tiny(seed=s) for s in range(2, 6)] + [
    workloads.random_small(seed=s, block_sizes=bs, num_requests=nr, max_ctx=mc,
                           max_chunk=ch, window=win)
    for s, bs, nr, mc, ch, win in [
        (20, (16,), 300, 2000, 400, 0),      # several CTAs, ragged tail
        (21, (32, 16), 200, 5000, 900, 0),
        (22, (1,), 50, 60, 30, 0),
        (23, (7, 16, 3), 90, 700, 200, 96),
        (24, (16,), 1, 100, 50, 0),          # a single request
        (25, (64,), 513, 3000, 5, 0),        # n not a multiple of 4
        (26, (1, 2, 3, 4, 5, 7, 16, 64), 90, 500, 80, 40),   # PKV_MAX_GROUPS groups
    ]] + [
    workloads.decode_heavy(seed=7, num_requests=40, max_ctx=192, pool=1024),   # W = 12
    workloads.decode_heavy(seed=8, num_requests=900, max_ctx=128, pool=8192),  # W = 8
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: f"{w.name}-{w.seed}")
def test_prepare_parity_small(wl):
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, len(wl.groups))
    # the call leaves the state as it was: a second call gives the same batch
    batch2, _, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch2, ref, len(wl.groups))
    assert st.get_error() == 0
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
def test_prepare_parity_full_size(make):
    """The five configurations at full size: every output element."""
    wl = make()
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, len(wl.groups))
    assert st.get_error() == 0
    st.close()
    orc.close()


def test_state_rows_match_oracle():
    """Churn of adds, updates and removes: every row's counters, token ids and
    block-table lines match the oracle's state model."""
    rng = np.random.default_rng(7)
    groups = [(16, 6, 500), (4, 20, 300)]
    st = pkv.State(12, 80, groups)
    orc = oracle.OracleState(12, 80, groups)
    live = []
    for step in range(400):
        op = rng.uniform()
        if (op < 0.45 or not live) and len(live) < 12:
            nt = int(rng.integers(0, 40))
            toks = rng.integers(0, 1000, nt)
            nc = int(rng.integers(0, nt + 1))
            b0 = rng.integers(0, 500, int(rng.integers(0, 4)))
            b1 = rng.integers(0, 300, int(rng.integers(0, 8)))
            r1 = st.add_request(toks, nc, [b0, b1])
            r2 = orc.add_request(toks, nc, [b0, b1])
            assert r1 == r2
            live.append(r1)
        elif op < 0.75 and live:
            r = live[int(rng.integers(0, len(live)))]
            nt = int(rng.integers(0, 5))
            toks = rng.integers(0, 1000, nt)
            info = st.row_info(r)
            b0 = rng.integers(0, 500, int(rng.integers(0, 2)))
            b1 = rng.integers(0, 300, int(rng.integers(0, 3)))
            nc = int(rng.integers(-1, info["n_tokens"] + nt + 1))
            rc1 = st.update_request(r, [b0, b1], toks, nc, check=False)
            rc2 = orc.update_request(r, [b0, b1], toks, nc, check=False)
            assert (rc1 == pkv.OK) == (rc2 == oracle.OK), (rc1, rc2)
        elif live:
            r = live.pop(int(rng.integers(0, len(live))))
            st.remove_request(r)
            orc.remove_request(r)
    for r in range(12):
        a = orc.read_row(r)
        info = st.row_info(r)
        assert info["active"] == a["active"]
        assert info["completed"] == a["completed"]
        b = st.read_row(r)
        assert b["completed"] == a["completed"]
        if a["active"]:
            assert b["tokens"].tolist() == a["tokens"].tolist()
        for g in range(2):
            assert b["block_table"][g].tolist() == a["block_table"][g].tolist()
            assert info["num_blocks"][g] == a["num_blocks"][g]
    st.close()


def test_long_token_arrays_over_several_ring_pieces():
    """With a 64 KiB staging ring (pieces of 4096 token ids), a 10000-token
    prompt and a 9000-token append are staged in pieces; the rows read back as
    the oracle's, and a batch over them is the oracle's batch."""
    rng = np.random.default_rng(31)
    groups = [(16, 1300, 3000)]
    L = 20100
    st = pkv.State(4, L, groups, ring_bytes=64 << 10)
    orc = oracle.OracleState(4, L, groups)
    toks = rng.integers(0, 128000, 10000)
    blocks = [rng.permutation(3000)[:1200].astype(np.int32)]
    r = st.add_request(toks, 9000, blocks)
    assert orc.add_request(toks, 9000, blocks) == r
    more = rng.integers(0, 128000, 9000)
    assert st.update_request(r, None, more, -1) == pkv.OK
    assert orc.update_request(r, None, more, -1) == oracle.OK
    a, b = orc.read_row(r), st.read_row(r)
    assert b["completed"] == a["completed"] == 9000
    np.testing.assert_array_equal(b["tokens"], a["tokens"])
    np.testing.assert_array_equal(b["block_table"][0], a["block_table"][0])
    rows, ns = np.array([r], np.int32), np.array([1000], np.int32)
    compare_batch(st.prepare_batch(rows, ns), orc.prepare_batch(rows, ns), 1)
    assert st.get_error() == 0
    st.close()


def test_advance_matches_oracle():
    wl = workloads.random_small(seed=31, num_requests=40, max_ctx=300, max_chunk=60)
    # room for every request to run its count a second time
    wl.max_model_len += 60
    for spec in wl.groups:
        spec.max_blocks_per_req += -(-60 // spec.block_size) + 1
    st, orc, rows = build_states(wl)
    reqs = wl.requests()
    # extend every request so it can run the same count again after advancing
    for h, c in wl.schedule:
        r = reqs[h]
        extra = np.arange(c, dtype=np.int32) + 11
        nb = []
        for spec, blk in zip(wl.groups, r.blocks):
            end = len(r.token_ids) + c
            k = max(0, -(-(end - len(blk) * spec.block_size) // spec.block_size))
            nb.append(np.arange(k, dtype=np.int32) % spec.num_blocks)
        st.update_request(rows[h], nb, extra)
        orc.update_request(rows[h], nb, extra)
    b1, r1, _, _ = prepare_both(st, orc, wl, rows, flags=pkv.ADVANCE)
    compare_batch(b1, r1, len(wl.groups))
    b2, r2, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(b2, r2, len(wl.groups))
    for h, c in wl.schedule:
        assert st.row_info(rows[h])["completed"] == reqs[h].num_computed + c
        assert st.read_row(rows[h], n_tokens=0)["completed"] == reqs[h].num_computed + c
    st.close()


def test_device_schedule_matches_host_schedule():
    wl = workloads.mixed_prefill(seed=3, rows=256)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    d_rows = torch.tensor(r, dtype=torch.int32, device="cuda")
    d_ns = torch.tensor(ns, dtype=torch.int32, device="cuda")
    batch = st.prepare_batch_device(d_rows, d_ns, int(ns.sum()))
    compare_batch(batch, ref, 1)
    # an unaligned device schedule (views offset by one element) works too
    d_rows2 = torch.zeros(len(r) + 1, dtype=torch.int32, device="cuda")
    d_ns2 = torch.zeros(len(r) + 1, dtype=torch.int32, device="cuda")
    d_rows2[1:] = d_rows
    d_ns2[1:] = d_ns
    batch = st.prepare_batch_device(d_rows2[1:], d_ns2[1:], int(ns.sum()))
    compare_batch(batch, ref, 1)
    assert st.get_error() == 0
    # with PKV_SCHEDULE_SETTLED (the schedule read before the previous kernel
    # ends), behind a long kernel that writes neither the schedule nor the
    # state, and with live tables too
    busy = torch.empty(1 << 27, dtype=torch.int32, device="cuda")
    busy.fill_(1)
    batch = st.prepare_batch_device(d_rows, d_ns, int(ns.sum()), flags=pkv.SCHEDULE_SETTLED)
    busy.fill_(2)
    batch2 = st.prepare_batch_device(d_rows, d_ns, int(ns.sum()),
                                     flags=pkv.SCHEDULE_SETTLED | pkv.LIVE_TABLES)
    compare_batch(batch, ref, 1)
    assert st.get_error() == 0
    for k in range(len(r)):
        live = -(-int(to_np(batch.seq_lens)[k]) // wl.groups[0].block_size)
        assert (to_np(batch2.block_tables[0])[k][:live] == ref["block_tables"][0][k][:live]).all()
    del busy
    st.close()


@pytest.mark.parametrize("n", [1, 32, 33, 256, 257])
def test_host_schedule_tiers(n):
    """Host schedules of up to 32 and up to 256 requests travel in the
    kernel's parameters (two block sizes), larger ones through the staging
    ring; both sides of each switch, two groups with block sizes 16 and 5,
    against the oracle."""
    wl = workloads.random_small(seed=300 + n, num_requests=n, block_sizes=(16, 5),
                                max_ctx=160, max_chunk=24, decode_frac=0.6)
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, 2)
    assert st.get_error() == 0
    st.close()


def test_large_host_schedules_back_to_back():
    """Host schedules of more than 256 requests are staged by a copy stream
    into two buffers used in turn: eight different schedules prepared back to
    back with no synchronisation in between, each into its own outputs, all
    equal the oracle's (a buffer reused too early would corrupt an earlier
    call's batch)."""
    wl = workloads.random_small(seed=71, num_requests=700, max_ctx=120, max_chunk=20,
                                decode_frac=0.7)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    rng = np.random.default_rng(72)
    subsets = [np.sort(rng.choice(len(r), int(rng.integers(257, len(r) + 1)), replace=False))
               for _ in range(8)]
    batches = [st.prepare_batch(r[idx], ns[idx]) for idx in subsets]
    torch.cuda.synchronize()
    for idx, batch in zip(subsets, batches):
        compare_batch(batch, orc.prepare_batch(r[idx], ns[idx]), 1)
    assert st.get_error() == 0
    st.close()


def test_prepare_host_call_reuses_buffers():
    """PrepareHostCall: the output struct marshalled once, schedules of any
    size up to the buffers' capacity, each against the oracle."""
    wl = workloads.mixed_prefill(seed=5, rows=256)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    out = st.alloc_batch(len(r), int(ns.sum()))
    call = pkv.PrepareHostCall(st, out)
    for k in (len(r), len(r) // 2, 1):
        sub_r, sub_ns = r[:k], ns[:k]
        batch = call(sub_r, sub_ns)
        compare_batch(batch, orc.prepare_batch(sub_r, sub_ns), 1)
    with pytest.raises(ValueError):
        call(np.concatenate([r, r[:1]]), np.concatenate([ns, ns[:1]]))
    assert st.get_error() == 0
    st.close()


def test_unaligned_block_table_output():
    wl = workloads.decode_heavy(seed=4, num_requests=50, max_ctx=640, pool=4096)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    n, W, T = len(r), wl.groups[0].max_blocks_per_req, int(ns.sum())
    out = st.alloc_batch(n, T)
    backing = torch.empty(n * W + 1, dtype=torch.int32, device="cuda")
    out.block_tables[0] = backing[1:].view(n, W)    # 4-byte aligned only
    st.prepare_batch(r, ns, out=out)
    compare_batch(out, ref, 1)
    st.close()


def test_empty_and_max_batches():
    st = pkv.State(pkv.MAX_BATCH, 64, [(16, 4, 70000)])
    b = st.prepare_batch([], [])
    assert b.total_tokens == 0 and to_np(b.query_start_loc).tolist() == [0]
    st.close()
    wl = workloads.random_small(seed=41, num_requests=pkv.MAX_BATCH, max_ctx=64,
                                max_chunk=8, decode_frac=0.8, rows=pkv.MAX_BATCH,
                                churn=False)
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, 1)
    assert st.get_error() == 0
    st.close()


def test_counts_above_the_packed_key_range():
    """A request running more than 65535 tokens in one step: the kernel ranks
    by raw (count, index) pairs instead of packed keys.  Ties between equal
    large counts, equal small counts and decodes keep schedule order."""
    rng = np.random.default_rng(65536)
    bs, W = 64, 2200
    st = pkv.State(16, 140000, [(bs, W, 20000)])
    orc = oracle.OracleState(16, 140000, [(bs, W, 20000)])
    ids = iter(rng.permutation(20000).tolist())
    # (known tokens, computed tokens, tokens scheduled this step)
    reqs = [(70000, 0, 70000), (3, 0, 3), (500, 499, 1), (70001, 1, 70000), (3, 0, 3),
            (9000, 8999, 1), (65536, 0, 65536), (1, 0, 1)]
    rows = []
    for ntok, comp, _ in reqs:
        tok = rng.integers(0, 128000, ntok).astype(np.int32)
        blocks = [[next(ids) for _ in range(-(-ntok // bs))]]
        r = st.add_request(tok, comp, blocks)
        assert orc.add_request(tok, comp, blocks) == r
        rows.append(r)
    order = rng.permutation(len(reqs))
    r = np.array([rows[k] for k in order], np.int32)
    ns = np.array([reqs[k][2] for k in order], np.int32)
    batch = st.prepare_batch(r, ns)
    ref = orc.prepare_batch(r, ns)
    compare_batch(batch, ref, 1)
    d_batch = st.prepare_batch_device(torch.tensor(r, device="cuda"),
                                      torch.tensor(ns, device="cuda"), int(ns.sum()))
    compare_batch(d_batch, ref, 1)
    assert st.get_error() == 0
    st.close()


def test_host_validation_errors():
    st = pkv.State(4, 16, [(4, 3, 100)])
    a = st.add_request(list(range(6)), 4, [[1, 2]])
    b = st.add_request(list(range(9)), 8, [[3, 4]])
    assert st.prepare_batch([a], [3], check=False) == pkv.ERR_CAPACITY    # no token 6
    assert st.prepare_batch([b], [1], check=False) == pkv.ERR_CAPACITY    # no block 2
    assert st.prepare_batch([a, a], [1, 1], check=False) == pkv.ERR_INVALID_ARG
    assert st.prepare_batch([a], [0], check=False) == pkv.ERR_INVALID_ARG
    assert st.prepare_batch([3], [1], check=False) == pkv.ERR_NOT_ACTIVE
    assert st.prepare_batch([9], [1], check=False) == pkv.ERR_INVALID_ARG
    c = st.add_request(list(range(10)), 8, [[-1, 5, 6]])   # block 0 freed
    assert to_np(st.prepare_batch([c], [2]).slot_mapping[0]).tolist() == [24, 25]
    d = st.add_request([1], 0, [[]])
    assert d == 3
    assert st.add_request([1], 0, [[]], check=False) == pkv.ERR_FULL
    st.remove_request(c)
    assert st.add_request(list(range(10)), 2, [[-1, 5, 6]]) == c
    assert st.prepare_batch([c], [1], check=False) == pkv.ERR_CAPACITY    # freed block
    assert st.add_request([1], 0, [[5, -1]], check=False) == pkv.ERR_INVALID_ARG
    assert st.add_request([1], 0, [[100]], check=False) == pkv.ERR_INVALID_ARG
    assert st.add_request([1], 2, [[]], check=False) == pkv.ERR_INVALID_ARG
    assert st.update_request(c, [[1, 2]], [], check=False) == pkv.ERR_CAPACITY
    assert st.remove_request(7, check=False) == pkv.ERR_INVALID_ARG
    st.remove_request(b)
    assert st.remove_request(b, check=False) == pkv.ERR_NOT_ACTIVE
    assert st.update_request(b, None, [1], check=False) == pkv.ERR_NOT_ACTIVE
    assert st.get_error() == 0
    st.close()


def test_device_checks_flag_and_skip():
    """The device-schedule entry point checks its inputs in the kernel: bad
    counts write nothing, bad rows / missing blocks write -1 and set bits."""
    st = pkv.State(8, 32, [(4, 4, 50)])
    r0 = st.add_request(list(range(12)), 8, [[1, 2, 3]])
    r1 = st.add_request(list(range(12)), 6, [[4, 5]])
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    # counts that do not sum to T: nothing written, COUNT bit
    out = st.alloc_batch(2, 3)
    out.positions.fill_(-7)
    st.prepare_batch_device(dev([r0, r1]), dev([1, 1]), 3, out=out)
    assert st.get_error() == pkv.DEVERR_COUNT
    assert to_np(out.positions).tolist() == [-7, -7, -7]
    st.prepare_batch_device(dev([r0, r1]), dev([0, 3]), 3, out=out)
    assert st.get_error() == pkv.DEVERR_COUNT
    # a row outside the table
    b = st.prepare_batch_device(dev([r0, 99]), dev([1, 2]), 3)
    assert st.get_error() & pkv.DEVERR_ROW
    assert to_np(b.index_mapping).tolist() == [r0, -1]
    assert to_np(b.positions)[1:].tolist() == [-1, -1]
    assert to_np(b.block_tables[0])[1].tolist() == [-1] * 4
    # r1 at position 8 needs block 2, which it does not have
    b = st.prepare_batch_device(dev([r1]), dev([3]), 3)
    assert st.get_error() & pkv.DEVERR_BLOCK
    assert to_np(b.slot_mapping[0]).tolist() == [5 * 4 + 2, 5 * 4 + 3, -1]
    # the error word is cleared by reading it
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("seed,block_sizes,max_ctx,window", [
    (401, (16,), 200, 0),          # 20 requests x W 13..15: the one-CTA small-batch kernel
    (402, (1,), 1000, 0),          # 20 requests x W 1000..1002 entries: over the small kernel's limit
    (403, (3, 16), 600, 64),       # two groups, a sliding window: small kernel
    (404, (1, 5), 1200, 256),      # two groups, over the limit
    (405, (1, 2, 3, 4, 5, 7, 16, 64), 150, 24),   # PKV_MAX_GROUPS groups: small kernel
    (406, (1, 2, 3, 4, 5, 7, 16, 64), 900, 0),    # PKV_MAX_GROUPS groups, over the limit
])
def test_small_batch_kernels(seed, block_sizes, max_ctx, window):
    """Batches of at most 32 requests whose table rows are small take the
    one-CTA kernel (sort in one warp); others the general one.  Both, on the
    host and the device schedule path, full and live tables, against the
    oracle."""
    wl = workloads.random_small(seed=seed, num_requests=20, block_sizes=block_sizes,
                                max_ctx=max_ctx, max_chunk=60, window=window)
    st, orc, rows = build_states(wl)
    G = len(wl.groups)
    batch, ref, r, ns = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, G)
    d_rows = torch.tensor(r, dtype=torch.int32, device="cuda")
    d_ns = torch.tensor(ns, dtype=torch.int32, device="cuda")
    compare_batch(st.prepare_batch_device(d_rows, d_ns, int(ns.sum())), ref, G)
    live = st.prepare_batch_device(d_rows, d_ns, int(ns.sum()), flags=pkv.LIVE_TABLES)
    for g in range(G):
        bs = wl.groups[g].block_size
        for k, sl in enumerate(ref["seq_lens"]):
            m = min(-(-int(sl) // bs), wl.groups[g].max_blocks_per_req)
            assert (to_np(live.block_tables[g])[k][:m] == ref["block_tables"][g][k][:m]).all()
    assert st.get_error() == 0
    st.close()


def test_device_schedule_repeated_row():
    """One batch row per request ("Extracting the Execution Batch from Global
    State"): a device schedule that lists a row twice keeps one listing (the
    one whose claim on the row lands first); the other is ranked as usual but
    all its outputs are -1, so no two tokens share a slot, and PKV_DEVERR_DUP
    is set.  The next call, without the repeat, is clean (a call's claims do
    not reach the next call)."""
    st = pkv.State(8, 32, [(4, 4, 50)])
    r0 = st.add_request(list(range(12)), 8, [[1, 2, 3]])
    r1 = st.add_request(list(range(12)), 6, [[4, 5]])
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    b = st.prepare_batch_device(dev([r0, r1, r0]), dev([1, 2, 1]), 4)
    assert st.get_error() == pkv.DEVERR_DUP
    # ascending counts, ties in schedule order: the two listings of r0, then r1
    im = to_np(b.index_mapping).tolist()
    assert im in ([r0, -1, r1], [-1, r0, r1])
    keep, rep = (0, 1) if im[0] == r0 else (1, 0)
    assert to_np(b.query_start_loc).tolist() == [0, 1, 2, 4]
    sl, pos = to_np(b.seq_lens).tolist(), to_np(b.positions).tolist()
    slots = to_np(b.slot_mapping[0]).tolist()
    assert sl[keep] == 9 and sl[rep] == -1 and sl[2] == 8
    assert pos[keep] == 8 and pos[rep] == -1 and pos[2:] == [6, 7]
    assert slots[keep] == 3 * 4 + 0 and slots[rep] == -1 and slots[2:] == [5 * 4 + 2, 5 * 4 + 3]
    assert to_np(b.block_tables[0])[rep].tolist() == [-1] * 4
    assert to_np(b.block_tables[0])[keep].tolist() == [1, 2, 3, -1]
    b = st.prepare_batch_device(dev([r1, r0]), dev([2, 1]), 3)
    assert st.get_error() == 0
    assert to_np(b.index_mapping).tolist() == [r0, r1]
    st.close()


def test_device_schedule_repeated_rows_large():
    """The same in a large schedule: of every row's listings exactly one keeps
    its outputs and the others get -1; the kept listings' outputs equal the
    oracle's batch of the kept listings alone."""
    wl = workloads.mixed_prefill(seed=8, rows=512)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    rng = np.random.default_rng(5)
    extra = rng.choice(len(r), 9, replace=False)
    r2 = np.concatenate([r, r[extra]])
    ns2 = np.concatenate([ns, np.ones(9, np.int32)])
    perm = rng.permutation(len(r2))
    r2, ns2 = r2[perm], ns2[perm]
    T = int(ns2.sum())
    b = st.prepare_batch_device(torch.tensor(r2, dtype=torch.int32, device="cuda"),
                                torch.tensor(ns2, dtype=torch.int32, device="cuda"), T)
    assert st.get_error() == pkv.DEVERR_DUP
    order = sorted(range(len(r2)), key=lambda i: (int(ns2[i]), i))
    rank_of = {i: k for k, i in enumerate(order)}
    im = to_np(b.index_mapping)
    qsl = to_np(b.query_start_loc)
    pos = to_np(b.positions)
    kept = [i for i in range(len(r2)) if im[rank_of[i]] >= 0]
    assert sorted(int(r2[i]) for i in kept) == sorted(set(int(x) for x in r2))
    for i in range(len(r2)):
        k = rank_of[i]
        if im[k] >= 0:
            assert im[k] == r2[i]
        else:
            assert (pos[qsl[k]:qsl[k + 1]] == -1).all()
            assert (to_np(b.block_tables[0])[k] == -1).all()
    ref = orc.prepare_batch(r2[kept], ns2[kept])
    got_rank = {int(r2[i]): rank_of[i] for i in kept}
    for kb, row in enumerate(ref["index_mapping"]):
        k = got_rank[int(row)]
        a0, a1 = qsl[k], qsl[k + 1]
        e0, e1 = ref["query_start_loc"][kb], ref["query_start_loc"][kb + 1]
        assert (pos[a0:a1] == ref["positions"][e0:e1]).all()
        assert (to_np(b.slot_mapping[0])[a0:a1] == ref["slot_mapping"][0][e0:e1]).all()
        assert (to_np(b.block_tables[0])[k] == ref["block_tables"][0][kb]).all()
    st.close()


LIVE_CASES = [
    lambda: workloads.mixed_prefill(seed=5, rows=256),
    lambda: workloads.two_groups(seed=6, num_requests=300, max_ctx=9000, window=1024),
    lambda: workloads.random_small(seed=42, block_sizes=(3, 16), num_requests=70,
                                   max_ctx=900, max_chunk=60),
    lambda: workloads.large_step(seed=3),
]


@pytest.mark.parametrize("make", LIVE_CASES, ids=["mixed", "two_groups", "odd_bs", "large"])
def test_live_tables_match_oracle(make):
    """PKV_LIVE_TABLES: every other output as before; of each gathered row, the
    live entries j < ceil(seq_len / bs) equal the oracle's; host and device
    schedule paths."""
    wl = make()
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    d_r = torch.tensor(r, dtype=torch.int32, device="cuda")
    d_n = torch.tensor(ns, dtype=torch.int32, device="cuda")
    for batch in (st.prepare_batch(r, ns, flags=pkv.LIVE_TABLES),
                  st.prepare_batch_device(d_r, d_n, int(ns.sum()), flags=pkv.LIVE_TABLES)):
        for key in ("index_mapping", "query_start_loc", "seq_lens", "positions", "input_ids"):
            np.testing.assert_array_equal(to_np(getattr(batch, key)), ref[key])
        for g, spec in enumerate(wl.groups):
            np.testing.assert_array_equal(to_np(batch.slot_mapping[g]), ref["slot_mapping"][g])
            got = to_np(batch.block_tables[g])
            for b, sl in enumerate(ref["seq_lens"]):
                live = min(-(-int(sl) // spec.block_size), spec.max_blocks_per_req)
                np.testing.assert_array_equal(got[b, :live], ref["block_tables"][g][b, :live])
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("width", [16, 17000])   # the one-CTA kernel, the general one
def test_device_schedule_position_past_the_model_length(width):
    """A device schedule (no host checks) whose request runs past the model
    length: its tokens at or past max_model_len get -1 positions, ids and
    slots and PKV_DEVERR_POSITION is set; the tokens before stay right."""
    st = pkv.State(8, 32, [(4, width, 50)])
    r = st.add_request(list(range(32)), 30, [list(range(8))])
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    b = st.prepare_batch_device(dev([r]), dev([4]), 4)
    assert st.get_error() == pkv.DEVERR_POSITION
    assert to_np(b.positions).tolist() == [30, 31, -1, -1]
    assert to_np(b.input_ids).tolist() == [30, 31, -1, -1]
    assert to_np(b.slot_mapping[0]).tolist() == [7 * 4 + 2, 7 * 4 + 3, -1, -1]
    assert to_np(b.seq_lens).tolist() == [34]
    st.close()
