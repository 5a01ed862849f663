"""pkv_apply_step (a whole step's scheduler output in one kernel) against the
oracle applying the same frees, adds and updates one call at a time."""
import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests.gpu_helpers import compare_batch

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def _compare_rows(st, orc, rows, G):
    for r in range(rows):
        a = orc.read_row(r)
        info = st.row_info(r)
        assert info["active"] == a["active"], r
        assert info["completed"] == a["completed"], r
        b = st.read_row(r)
        assert b["completed"] == a["completed"], r
        if a["active"]:
            assert info["n_tokens"] == len(a["tokens"]), r
            assert b["tokens"].tolist() == a["tokens"].tolist(), r
        for g in range(G):
            assert b["block_table"][g].tolist() == a["block_table"][g].tolist(), (r, g)
            assert info["num_blocks"][g] == a["num_blocks"][g], (r, g)


def _packed(finished, new, cached, G):
    """The same scheduler output as int32 CSR arrays (apply_step_arrays)."""
    def csr(lists):
        off = np.zeros(len(lists) + 1, np.int32)
        off[1:] = np.cumsum([len(x) for x in lists])
        flat = np.concatenate([np.asarray(x, np.int32) for x in lists]) if off[-1] else \
            np.zeros(0, np.int32)
        return off, flat
    nt, ct = csr([x[0] for x in new]), csr([x[1] for x in cached])
    nb = [csr([x[2][g] for x in new]) for g in range(G)]
    cb = [csr([x[3][g] for x in cached]) for g in range(G)]
    return (np.asarray(finished, np.int32), nt[0], nt[1], [x[1] for x in new],
            [b[0] for b in nb], [b[1] for b in nb], [x[0] for x in cached], ct[0], ct[1],
            [x[2] for x in cached], [b[0] for b in cb], [b[1] for b in cb])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_apply_step_matches_sequential_calls(seed):
    """Even steps through apply_step (Python lists), odd steps through
    apply_step_arrays (the same output packed as CSR arrays)."""
    rng = np.random.default_rng(seed)
    groups = [(16, 12, 4000), (4, 40, 3000)]
    R, L = 48, 160
    st = pkv.State(R, L, groups, ring_bytes=1 << 20)   # small ring: several pieces
    orc = oracle.OracleState(R, L, groups)
    live = {}   # row -> (n_tokens, nblk per group)
    for step in range(60):
        rows = list(live)
        rng.shuffle(rows)
        nf = int(rng.integers(0, min(len(rows), 6) + 1))
        finished = rows[:nf]
        free_after = R - len(live) + nf
        new = []
        for _ in range(int(rng.integers(0, min(free_after, 8) + 1))):
            nt = int(rng.integers(0, 120))
            toks = rng.integers(0, 1000, nt)
            nc = int(rng.integers(0, nt + 1))
            b0 = rng.integers(0, 4000, int(rng.integers(0, 8)))
            nb1 = int(rng.integers(0, 30))
            lead = int(rng.integers(0, nb1 + 1)) if rng.uniform() < 0.3 else 0
            b1 = np.concatenate([np.full(lead, -1), rng.integers(0, 3000, nb1 - lead)])
            new.append((toks, nc, [b0, b1]))
        cached = []
        for r in rows[nf:]:
            if rng.uniform() < 0.6:
                nt, (n0, n1) = live[r]
                k = int(rng.integers(0, min(4, L - nt) + 1))
                m0 = int(rng.integers(0, min(2, 12 - n0) + 1))
                m1 = int(rng.integers(0, min(3, 40 - n1) + 1))
                nc = int(rng.integers(-1, nt + k + 1))
                cached.append((r, rng.integers(0, 1000, k), nc,
                               [rng.integers(0, 4000, m0), rng.integers(0, 3000, m1)]))
        if step % 2 == 0:
            got = st.apply_step(finished, new, cached)
        else:
            got = st.apply_step_arrays(*_packed(finished, new, cached, 2)).tolist()
        for r in finished:
            orc.remove_request(r)
            del live[r]
        want = [orc.add_request(t, nc, b) for t, nc, b in new]
        assert got == want
        for (t, nc, b), r in zip(new, got):
            live[r] = (len(t), (len(b[0]), len(b[1])))
        for r, t, nc, b in cached:
            orc.update_request(r, b, t, nc)
            nt, (n0, n1) = live[r]
            live[r] = (nt + len(t), (n0 + len(b[0]), n1 + len(b[1])))
        if step % 15 == 14:
            _compare_rows(st, orc, R, 2)
    _compare_rows(st, orc, R, 2)
    assert st.get_error() == 0
    st.close()


def test_apply_step_validates_as_a_whole():
    st = pkv.State(4, 32, [(4, 4, 100)])
    a = st.add_request(list(range(8)), 2, [[1, 2]])
    b = st.add_request(list(range(8)), 2, [[3]])
    before = [st.read_row(r) for r in (a, b)]
    # the update of b overflows the table row: nothing of the step happens
    rc = st.apply_step(finished=[a], new=[([5, 6], 0, [[7]])],
                       cached=[(b, [9], -1, [[4, 5, 6, 7]])], check=False)
    assert rc == pkv.ERR_CAPACITY
    assert st.row_info(a)["active"] and st.row_info(b)["active"]
    after = [st.read_row(r) for r in (a, b)]
    for x, y in zip(before, after):
        assert x["tokens"].tolist() == y["tokens"].tolist()
        assert x["block_table"][0].tolist() == y["block_table"][0].tolist()
    assert st.apply_step(finished=[a, a], check=False) == pkv.ERR_INVALID_ARG
    assert st.apply_step(cached=[(b, [], -1, [[]]), (b, [], -1, [[]])],
                         check=False) == pkv.ERR_INVALID_ARG
    assert st.apply_step(finished=[a], cached=[(a, [], -1, [[]])],
                         check=False) == pkv.ERR_NOT_ACTIVE
    assert st.apply_step(new=[([1], 0, [[]])] * 3, check=False) == pkv.ERR_FULL
    # freeing a row lets a new request of the same step reuse it
    assert st.apply_step(finished=[a], new=[([1, 2, 3], 1, [[9]])] * 3) == [0, 2, 3]
    assert st.read_row(0)["block_table"][0].tolist() == [9, -1, -1, -1]
    st.close()


def test_batch_after_applied_steps_matches_oracle():
    """A workload built through pkv_apply_step prepares the same batch as the
    oracle built through individual calls."""
    wl = workloads.mixed_prefill(seed=12, rows=256, budget=3000, num_decode=40)
    G = len(wl.groups)
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    orc = oracle.OracleState(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows_o = workloads.apply_ops(orc, wl)
    rows_l = {}
    # replay the same program, one step per block of consecutive adds/removes
    pending_new, pending_fin = [], []

    def flush():
        got = st.apply_step(finished=[rows_l.pop(h) for h in pending_fin],
                            new=[(r.token_ids, r.num_computed, r.blocks) for r in pending_new])
        for r, row in zip(pending_new, got):
            rows_l[r.handle] = row
        pending_new.clear()
        pending_fin.clear()

    for op in wl.ops:
        if op[0] == "add":
            pending_new.append(op[1])
        else:
            if pending_new:
                flush()
            pending_fin.append(op[1])
    flush()
    assert rows_l == rows_o
    r, ns = workloads.schedule_arrays(wl, rows_l)
    compare_batch(st.prepare_batch(r, ns), orc.prepare_batch(r, ns), G)
    st.close()
