"""pkv_prepare_batch_static, the batch build that allocates no device memory,
against the regular host-schedule entry point pkv_prepare_batch.

Callers that cannot allocate -- an engine that has handed all free HBM to its
KV cache, a plugin running inside another runtime, code without a pkv_state --
keep the request-state table in their own device arrays and call the static
variant, whose only scratch (the staged schedule) is a fixed array inside the
library.  Here that table is built by hand as a caller would, in the layout
pkv_state keeps, and both entry points must give bit-identical batches on two
calls in a row (the second call reusing the array the first one filled).

This file is named to be collected last."""
import ctypes as C

import numpy as np
import pytest

import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from paged_kv_prep_gb300._lib import BatchOut, GroupSpec, lib

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def caller_table(wl, rows):
    """The request-state table in caller-owned device memory."""
    R, L = wl.max_reqs, wl.max_model_len
    completed = np.zeros(R, np.int32)
    tokens = np.zeros((R, L), np.int32)
    tables = [np.full((R, g.max_blocks_per_req), -1, np.int32) for g in wl.groups]
    for h, req in wl.requests().items():
        if h not in rows:
            continue
        r = rows[h]
        completed[r] = req.num_computed
        tokens[r, :len(req.token_ids)] = req.token_ids
        for g, blocks in enumerate(req.blocks):
            tables[g][r, :len(blocks)] = blocks
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    return dev(completed), dev(tokens), [dev(t) for t in tables]


def call_static(wl, table, rows, ns, out, d_err):
    completed, tokens, tables = table
    G = len(wl.groups)
    specs = (GroupSpec * G)(*[GroupSpec(g.block_size, g.max_blocks_per_req, g.num_blocks)
                              for g in wl.groups])
    tptrs = (C.c_void_p * G)(*[t.data_ptr() for t in tables])
    r = np.ascontiguousarray(rows, np.int32)
    c = np.ascontiguousarray(ns, np.int32)
    st = out.struct()
    total = C.c_int32(-1)
    rc = lib().pkv_prepare_batch_static(
        C.c_void_p(completed.data_ptr()), C.c_void_p(tokens.data_ptr()), wl.max_reqs,
        wl.max_model_len, G, specs, tptrs, r.ctypes.data_as(C.POINTER(C.c_int32)),
        c.ctypes.data_as(C.POINTER(C.c_int32)), len(r), C.byref(st),
        C.c_void_p(d_err.data_ptr()), C.byref(total),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, total.value


def assert_same(a, b, groups):
    for name in ("index_mapping", "query_start_loc", "seq_lens", "positions", "input_ids"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    for g in range(groups):
        assert torch.equal(a.block_tables[g], b.block_tables[g]), g
        assert torch.equal(a.slot_mapping[g], b.slot_mapping[g]), g


@pytest.mark.parametrize("name,kw", [
    ("mixed_prefill", dict(rows=512)),
    ("two_groups", dict(num_requests=600, max_ctx=8192, window=1024)),
    ("decode_heavy", dict(num_requests=300, max_ctx=4096)),   # every count 1
    ("tiny", {}),                                             # the one-CTA kernel
])
def test_static_variant_matches_regular_entry_point(name, kw):
    wl = workloads.build(name, seed=9, **kw)
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows = workloads.apply_ops(st, wl)
    table = caller_table(wl, rows)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r, ns = workloads.schedule_arrays(wl, rows)
    # two calls in a row: the full schedule, then a different, smaller one in
    # another order, which must not see anything the first call left behind
    rng = np.random.default_rng(3)
    pick = rng.permutation(len(r))[: max(1, len(r) // 3)]
    for rr, nn in ((r, ns), (r[pick], ns[pick])):
        want = st.prepare_batch(rr, nn)
        got = st.alloc_batch(len(rr), int(nn.sum()))
        for t in (got.index_mapping, got.query_start_loc, got.seq_lens, got.positions,
                  got.input_ids, *got.block_tables, *got.slot_mapping):
            t.fill_(-7)
        rc, total = call_static(wl, table, rr, nn, got, d_err)
        assert rc == pkv.OK
        assert total == int(nn.sum())
        torch.cuda.synchronize()
        assert_same(got, want, len(wl.groups))
    assert int(d_err.item()) == 0
    # more requests than the fixed array holds are refused
    big = np.zeros(pkv._lib.STATIC_MAX_BATCH + 1, np.int32)
    out = st.alloc_batch(1, 1)
    wl_big = workloads.Workload("x", 0, pkv._lib.STATIC_MAX_BATCH + 1, 4, wl.groups, 1, 1,
                                "float16", 1)
    rc, _ = call_static(wl_big, table, big, big + 1, out, d_err)
    assert rc == pkv.ERR_INVALID_ARG
    st.close()


def _pinned(a):
    t = torch.from_numpy(np.ascontiguousarray(a, np.int32)).pin_memory()
    return t, t.numpy()


@pytest.mark.parametrize("count", [200, 700])
def test_static_pinned_arrays_reused_at_once(count):
    """A scheduler that keeps its output in page-locked memory may overwrite
    rows and num_sched as soon as the call returns, even while earlier GPU
    work delays the batch build: up to 256 requests ride in the kernel's
    parameters, more are copied out of the caller's arrays before the call
    returns."""
    wl = workloads.build("two_groups", seed=11, num_requests=800, max_ctx=4096, window=1024)
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows = workloads.apply_ops(st, wl)
    table = caller_table(wl, rows)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r, ns = workloads.schedule_arrays(wl, rows)
    r, ns = r[:count], ns[:count]
    want = st.prepare_batch(r, ns)
    torch.cuda.synchronize()
    keep_r, pr = _pinned(r)
    keep_n, pn = _pinned(ns)
    got = st.alloc_batch(len(r), int(ns.sum()))
    # queue about a millisecond of unrelated work first
    busy = torch.empty(1 << 28, dtype=torch.int32, device="cuda")
    for _ in range(4):
        busy.fill_(3)
    rc, total = call_static(wl, table, pr, pn, got, d_err)
    assert rc == pkv.OK and total == int(ns.sum())
    pr[:] = pr[::-1].copy()       # reuse both arrays at once
    pn[:] = 1
    torch.cuda.synchronize()
    assert_same(got, want, len(wl.groups))
    assert int(d_err.item()) == 0
    del busy, keep_r, keep_n
    st.close()


def test_static_empty_repeated_and_captured():
    wl = workloads.build("mixed_prefill", seed=4, rows=512)
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows = workloads.apply_ops(st, wl)
    table = caller_table(wl, rows)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r, ns = workloads.schedule_arrays(wl, rows)
    # n == 0: only query_start_loc[0] is written
    out = st.alloc_batch(0, 0)
    out.query_start_loc.fill_(-7)
    rc, total = call_static(wl, table, r[:0], ns[:0], out, d_err)
    torch.cuda.synchronize()
    assert rc == pkv.OK and total == 0
    assert out.query_start_loc.tolist() == [0]
    # a row listed twice is refused before anything runs
    rr = np.concatenate([r, r[:1]])
    nn = np.concatenate([ns, ns[:1]])
    out = st.alloc_batch(len(rr), int(nn.sum()))
    rc, _ = call_static(wl, table, rr, nn, out, d_err)
    assert rc == pkv.ERR_INVALID_ARG
    # more than 256 requests while the stream is being captured: refused
    many = np.arange(300, dtype=np.int32)
    ones = np.ones(300, np.int32)
    out = st.alloc_batch(300, 300)
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g.capture_begin()
        d_err.add_(0)
        rc, _ = call_static(wl, table, many, ones, out, d_err)
        g.capture_end()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert rc == pkv.ERR_INVALID_ARG
    assert int(d_err.item()) == 0
    st.close()
