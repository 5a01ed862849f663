"""Pure decode steps -- every scheduled request runs one token, so T == n and
the stable ascending sort keeps schedule order ("Extracting the Execution
Batch from Global State") -- take the batch build's decode kernel.  Against
the oracle, element by element: host schedules (in the launch parameters or
staged) and device schedules (aligned or not, settled or not), full and live
block tables, one to eight KV-cache groups, the no-allocation entry point.
Then its checks: a count other than 1 writes nothing, a repeated or unknown
row gets -1 outputs, a missing block or a position past the model length is
flagged."""
import numpy as np
import pytest

import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests.gpu_helpers import build_states, compare_batch, to_np
from tests.helpers import schedule_arrays

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def pure_decode(seed, n, block_sizes, max_ctx, window=0):
    wl = workloads.random_small(seed=seed, num_requests=n, block_sizes=block_sizes,
                                max_ctx=max_ctx, max_chunk=1, decode_frac=1.0, window=window)
    assert all(c == 1 for _, c in wl.schedule)
    return wl


def dev(a):
    return torch.tensor(np.asarray(a, np.int32), dtype=torch.int32, device="cuda")


def compare_live(batch, ref, wl):
    """Live tables: the entries attention reads, j < ceil(seq_len / bs)."""
    for g, spec in enumerate(wl.groups):
        got = to_np(batch.block_tables[g])
        for b, sl in enumerate(ref["seq_lens"]):
            k = min(-(-int(sl) // spec.block_size), spec.max_blocks_per_req)
            np.testing.assert_array_equal(got[b, :k], ref["block_tables"][g][b, :k])


CASES = [
    # seed, n, block sizes, max context, window
    (501, 1, (1,), 20000, 0),          # one request, a 20000-entry row
    (502, 20, (1,), 1000, 0),          # n <= 32 but rows too long for the one-CTA kernel
    (503, 33, (32, 16), 2000, 0),      # a host schedule in the 256-request parameter block
    (504, 256, (16,), 8192, 0),        # the decode-heavy shape
    (505, 257, (3, 16), 900, 64),      # a staged host schedule; a sliding window
    (506, 1001, (1, 64), 300, 0),      # n not a multiple of 4; one position per block
    (507, 600, (1, 2, 3, 4, 5, 7, 16, 64), 200, 40),   # eight groups
    (508, 5000, (16,), 20, 0),         # many requests of a one-entry row: 256 per CTA
    (509, 16384, (16, 4), 64, 0),      # PKV_MAX_BATCH requests
]


@pytest.mark.parametrize("seed,n,bss,max_ctx,window", CASES)
def test_pure_decode_matches_oracle(seed, n, bss, max_ctx, window):
    wl = pure_decode(seed, n, bss, max_ctx, window)
    st, orc, rows = build_states(wl)
    G = len(wl.groups)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    assert ref["query_start_loc"].tolist() == list(range(n + 1))
    compare_batch(st.prepare_batch(r, ns), ref, G)
    compare_live(st.prepare_batch(r, ns, flags=pkv.LIVE_TABLES), ref, wl)
    # device schedules: aligned, settled or not; then both arrays one int32
    # off a 16-byte boundary (no vector reads of the counts)
    d_r, d_n = dev(r), dev(ns)
    compare_batch(st.prepare_batch_device(d_r, d_n, n), ref, G)
    compare_batch(st.prepare_batch_device(d_r, d_n, n, flags=pkv.SCHEDULE_SETTLED), ref, G)
    compare_live(st.prepare_batch_device(d_r, d_n, n, flags=pkv.LIVE_TABLES), ref, wl)
    off_r = dev(np.concatenate([[0], r]))[1:]
    off_n = dev(np.concatenate([[0], ns]))[1:]
    compare_batch(st.prepare_batch_device(off_r, off_n, n), ref, G)
    assert st.get_error() == 0
    st.close()


def test_pure_decode_advance():
    """PKV_ADVANCE on a decode step moves every request's completed_tokens on
    by one; the batch itself is the one without the flag."""
    wl = pure_decode(520, 300, (16,), 500)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    before = [st.row_info(int(x))["completed"] for x in r]
    ref = orc.prepare_batch(r, ns, advance=True)
    compare_batch(st.prepare_batch(r, ns, flags=pkv.ADVANCE), ref, 1)
    torch.cuda.synchronize()
    assert [st.row_info(int(x))["completed"] for x in r] == [c + 1 for c in before]
    assert st.get_error() == 0
    st.close()


def test_pure_decode_count_errors_write_nothing():
    """T == n but a count is not 1 (so some count is < 1, or the counts do not
    sum to T): PKV_DEVERR_COUNT and no output written, as for any batch."""
    wl = pure_decode(521, 40, (16,), 500)
    st, orc, rows = build_states(wl)
    r, _ = schedule_arrays(wl, rows)
    out = st.alloc_batch(40, 41)
    for bad in ([1] * 38 + [0, 2], [1] * 39 + [2], [1] * 39 + [-1]):
        for t in (out.index_mapping, out.query_start_loc, out.seq_lens, out.positions,
                  out.input_ids, out.block_tables[0], out.slot_mapping[0]):
            t.fill_(-7)
        st.prepare_batch_device(dev(r), dev(bad), 40, out=out)
        assert st.get_error() == pkv.DEVERR_COUNT
        for t in (out.index_mapping, out.query_start_loc, out.seq_lens, out.positions,
                  out.input_ids, out.block_tables[0], out.slot_mapping[0]):
            assert (to_np(t) == -7).all()
    st.close()


def test_pure_decode_repeated_rows():
    """A device decode schedule listing rows more than once: of each row's
    listings exactly one keeps its outputs (those of the schedule without the
    repeats), every other one gets -1 everywhere, PKV_DEVERR_DUP is set; batch
    entry b is still schedule entry b."""
    wl = pure_decode(522, 300, (16, 32), 3000)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    where = {int(x): k for k, x in enumerate(r)}
    rr = np.concatenate([r[:150], r[[7]], r[150:], r[[100, 7]]]).astype(np.int32)
    m = len(rr)
    for flags in (0, pkv.SCHEDULE_SETTLED):
        b = st.prepare_batch_device(dev(rr), dev(np.ones(m, np.int32)), m, flags=flags)
        assert st.get_error() == pkv.DEVERR_DUP
        assert to_np(b.query_start_loc).tolist() == list(range(m + 1))
        im, sl = to_np(b.index_mapping), to_np(b.seq_lens)
        pos, ids = to_np(b.positions), to_np(b.input_ids)
        tabs = [to_np(t) for t in b.block_tables]
        slots = [to_np(s) for s in b.slot_mapping]
        for x, k in where.items():
            listings = np.flatnonzero(rr == x)
            kept = [e for e in listings if im[e] == x]
            assert len(kept) == 1, (x, listings, im[listings])
            e = kept[0]
            assert sl[e] == ref["seq_lens"][k] and pos[e] == ref["positions"][k]
            assert ids[e] == ref["input_ids"][k]
            for g in range(2):
                assert slots[g][e] == ref["slot_mapping"][g][k]
                np.testing.assert_array_equal(tabs[g][e], ref["block_tables"][g][k])
            for e in listings:
                if e == kept[0]:
                    continue
                assert im[e] == -1 and sl[e] == -1 and pos[e] == -1 and ids[e] == -1
                for g in range(2):
                    assert slots[g][e] == -1 and (tabs[g][e] == -1).all()
    # the next call, without the repeats, is clean
    compare_batch(st.prepare_batch_device(dev(r), dev(ns), len(r)), ref, 2)
    assert st.get_error() == 0
    st.close()


def test_pure_decode_bad_rows_positions_and_blocks():
    """Rows of 5000 entries, so four requests exceed the one-CTA kernel's
    limit: an unknown row (PKV_DEVERR_ROW), a position at the model length
    (PKV_DEVERR_POSITION) and a missing block (PKV_DEVERR_BLOCK) each get
    -1 where the method cannot give a value; the good request is unchanged."""
    st = pkv.State(8, 32, [(4, 5000, 50)])
    good = st.add_request(list(range(12)), 8, [[1, 2, 3]])      # position 8: block 3
    short = st.add_request(list(range(12)), 8, [[4, 5]])        # position 8 has no block
    full = st.add_request(list(range(32)), 32, [[6, 7, 8, 9]])  # position 32 = the model length
    b = st.prepare_batch_device(dev([good, 99, short, full]), dev([1, 1, 1, 1]), 4)
    err = st.get_error()
    assert err == pkv.DEVERR_ROW | pkv.DEVERR_BLOCK | pkv.DEVERR_POSITION
    assert to_np(b.index_mapping).tolist() == [good, -1, short, full]
    assert to_np(b.query_start_loc).tolist() == [0, 1, 2, 3, 4]
    assert to_np(b.seq_lens).tolist() == [9, -1, 9, 33]
    assert to_np(b.positions).tolist() == [8, -1, 8, -1]
    assert to_np(b.input_ids).tolist() == [8, -1, 8, -1]
    assert to_np(b.slot_mapping[0]).tolist() == [3 * 4 + 0, -1, -1, -1]
    tab = to_np(b.block_tables[0])
    assert tab[0, :4].tolist() == [1, 2, 3, -1] and (tab[0, 4:] == -1).all()
    assert (tab[1] == -1).all()
    assert tab[2, :3].tolist() == [4, 5, -1]
    assert tab[3, :5].tolist() == [6, 7, 8, 9, -1]
    st.close()


def test_pure_decode_full_size_decode_heavy_against_oracle():
    """The decode-heavy configuration at full size (256 decodes, 512-entry
    rows) through the device path as the bench runs it."""
    wl = workloads.decode_heavy(seed=0)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    for flags in (pkv.SCHEDULE_SETTLED, pkv.SCHEDULE_SETTLED | pkv.LIVE_TABLES):
        b = st.prepare_batch_device(dev(r), dev(ns), len(r), flags=flags)
        if flags & pkv.LIVE_TABLES:
            compare_live(b, ref, wl)
        else:
            compare_batch(b, ref, 1)
    assert st.get_error() == 0
    st.close()


def test_pure_decode_large_against_oracle():
    """4096 decodes with 4096-entry rows (134 MB of table rows), as `bench.py
    --workload decode_large` runs it: every output element against the
    oracle, full and live tables."""
    wl = workloads.build("decode_large", seed=0)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    d_r, d_n = dev(r), dev(ns)
    compare_batch(st.prepare_batch_device(d_r, d_n, len(r), flags=pkv.SCHEDULE_SETTLED), ref, 1)
    compare_live(st.prepare_batch_device(d_r, d_n, len(r),
                                         flags=pkv.SCHEDULE_SETTLED | pkv.LIVE_TABLES), ref, wl)
    compare_batch(st.prepare_batch(r, ns), ref, 1)
    assert st.get_error() == 0
    st.close()
