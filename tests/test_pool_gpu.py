"""allocate_slots / release_blocks on the GPU against the CPU oracle."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests.gpu_helpers import compare_batch

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def _same_state(st, orc, R, G):
    for g in range(G):
        assert st.pool_size(g) == len(orc.pool(g)), g
        np.testing.assert_array_equal(st.pool(g), orc.pool(g))
    for r in range(R):
        a = orc.read_row(r)
        if not a["active"]:
            continue
        b = st.read_row(r, n_tokens=0)
        info = st.row_info(r)
        for g in range(G):
            assert b["block_table"][g].tolist() == a["block_table"][g].tolist(), (r, g)
            assert info["num_blocks"][g] == a["num_blocks"][g], (r, g)


def test_pages_example_on_gpu():
    g = json.load(open(os.path.join(HERE, "golden", "prefix_cache_example.json")))
    bs, fx = g["block_size"], g["fixture_choices"]
    B = fx["system_prompt"] + fx["B_suffix"]
    st = pkv.State(8, 64, [(bs, 8, 100)])
    st.pool_reset(0, [70, 71, fx["B3"]])
    rb = st.add_request(B, 8, [[fx["P1"], fx["P2"]]])
    adm, nb = st.allocate_slots([rb], [len(B) - 8])
    pr = g["printed_on_the_pages"]
    assert adm == 1 and nb.tolist() == [[len(pr["B_newly_allocated"])]]
    assert st.read_row(rb)["block_table"][0][:3].tolist() == \
        [fx[name] for name in pr["B_logical_block_table"]]
    assert st.pool(0).tolist() == [70, 71]
    st.close()


def test_page_order_cases_on_gpu():
    """Step (2) frees precede the check of step (4): they serve the request
    itself and later requests of the call, and a refused request's frees
    stand (the oracle's pins, on the device path)."""
    # admitted on its own frees: takes 42
    st = pkv.State(4, 64, [(4, 8, 100)])
    st.pool_reset(0, [])
    r = st.add_request(list(range(24)), 20, [[40, 41, 42, 43, 44]])
    adm, nb = st.allocate_slots([r], [4], windows=[8])
    assert adm == 1 and nb.tolist() == [[1]]
    assert st.read_row(r)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, 42]
    assert st.pool(0).tolist() == [40, 41]
    assert st.row_info(r)["num_blocks"][0] == 6
    st.close()
    # one request's frees serve the next
    st = pkv.State(4, 64, [(4, 8, 100)])
    st.pool_reset(0, [])
    a = st.add_request(list(range(22)), 20, [[40, 41, 42, 43, 44, 45]])
    b = st.add_request(list(range(8)), 0, [[]])
    adm, nb = st.allocate_slots([a, b], [2, 8], windows=[8])
    assert adm == 2 and nb.tolist() == [[0], [2]]
    assert st.read_row(b)["block_table"][0][:3].tolist() == [42, 41, -1]
    assert st.pool(0).tolist() == [40]
    st.close()
    # refused, frees stand; a repeated row changes nothing
    st = pkv.State(4, 64, [(4, 12, 100)])
    st.pool_reset(0, [])
    r = st.add_request(list(range(40)), 20, [[40, 41, 42, 43, 44]])
    adm, nb = st.allocate_slots([r], [20], windows=[8])
    assert adm == 0 and nb.tolist() == [[0]]
    assert st.read_row(r)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, -1]
    assert st.pool(0).tolist() == [40, 41, 42]
    with pytest.raises(pkv.PkvError):
        st.allocate_slots([r, r], [1, 1], windows=[8])
    assert st.pool(0).tolist() == [40, 41, 42]
    # a request longer than its table row: an error, nothing moved
    with pytest.raises(pkv.PkvError):
        st.allocate_slots([r], [40], windows=[8])
    assert st.pool(0).tolist() == [40, 41, 42]
    assert st.read_row(r)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, -1]
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_allocate_and_release_match_oracle(seed):
    rng = np.random.default_rng(seed)
    R, L = 40, 600
    groups = [(16, 40, 900), (4, 160, 2500)]
    windows = [0, 48]
    st = pkv.State(R, L, groups)
    orc = oracle.OracleState(R, L, groups)
    for g, (_, _, nbk) in enumerate(groups):
        ids = rng.permutation(nbk)[: int(nbk * 0.8)].astype(np.int32)
        st.pool_reset(g, ids)
        orc.pool_reset(g, ids)
    live = []
    for rnd in range(40):
        # arrivals: a prompt with nothing allocated yet
        for _ in range(int(rng.integers(0, 4))):
            if len(live) >= R:
                break
            nt = int(rng.integers(1, 200))
            toks = rng.integers(0, 1000, nt)
            r1 = st.add_request(toks, 0, [[], []])
            r2 = orc.add_request(toks, 0, [[], []])
            assert r1 == r2
            live.append(r1)
        # a step: every live request asks for its next chunk or token
        rng.shuffle(live)
        rows, new, la = [], [], []
        for r in live:
            info = orc.read_row(r)
            room = L - info["completed"] - 4
            if room <= 0:
                continue
            k = int(rng.integers(1, min(room, 64) + 1))
            rows.append(r)
            new.append(k)
            la.append(int(rng.integers(0, 3)))
        wm = int(rng.integers(0, 4))
        got = st.allocate_slots(rows, new, la, windows, wm)
        want = orc.allocate_slots(rows, new, la, windows, wm)
        assert got[0] == want[0], rnd
        np.testing.assert_array_equal(got[1], want[1])
        # the admitted requests run their tokens (computed count advances)
        for r, k in zip(rows[:got[0]], new[:got[0]]):
            c = orc.read_row(r)["completed"]
            nt = len(orc.read_row(r)["tokens"])
            extra = max(0, c + k - nt)
            toks = rng.integers(0, 1000, extra)
            st.update_request(r, None, toks, c + k)
            orc.update_request(r, None, toks, c + k)
        # some requests finish and give their blocks back
        done = [r for r in live if rng.uniform() < 0.15]
        if done:
            st.release_blocks(done)
            orc.release_blocks(done)
            for r in done:
                st.remove_request(r)
                orc.remove_request(r)
                live.remove(r)
        if rnd % 10 == 9:
            _same_state(st, orc, R, 2)
    _same_state(st, orc, R, 2)
    st.close()


def test_batch_after_allocation_matches_oracle():
    """Blocks handed out by allocate_slots give the same prepared batch as the
    oracle's allocation."""
    rng = np.random.default_rng(9)
    R, L = 64, 2048
    groups = [(16, 128, 6000), (16, 128, 6000)]
    st = pkv.State(R, L, groups)
    orc = oracle.OracleState(R, L, groups)
    for g in range(2):
        ids = rng.permutation(6000).astype(np.int32)
        st.pool_reset(g, ids)
        orc.pool_reset(g, ids)
    rows, new = [], []
    for _ in range(R):
        nt = int(rng.integers(2, 1500))
        toks = rng.integers(0, 128000, nt)
        nc = int(rng.integers(0, nt))
        r = st.add_request(toks, nc, [[], []])
        orc.add_request(toks, nc, [[], []])
        rows.append(r)
        new.append(nt - nc)
    adm_l = st.allocate_slots(rows, new, windows=[0, 256])
    adm_o = orc.allocate_slots(rows, new, windows=[0, 256])
    assert adm_l[0] == adm_o[0] == R
    order = rng.permutation(R)
    r = np.array(rows, np.int32)[order]
    ns = np.array(new, np.int32)[order]
    compare_batch(st.prepare_batch(r, ns), orc.prepare_batch(r, ns), 2)
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("seed,windows,wm", [(3, [0, 40], 0), (4, [24, 0], 2), (5, [16, 64], 1)])
def test_large_batches_match_oracle(seed, windows, wm):
    """Thousands of requests per call, with window frees everywhere and pools
    small enough that most calls end in a refusal: pops reach back over many
    earlier requests (the pop kernel's walk), and deep pops take the ids the
    stack started with."""
    rng = np.random.default_rng(seed)
    R, L = 3000, 400
    groups = [(4, 100, 40000), (8, 50, 20000)]
    st = pkv.State(R, L, groups)
    orc = oracle.OracleState(R, L, groups)
    pools = []
    for g, (_, _, nbk) in enumerate(groups):
        ids = rng.permutation(nbk).astype(np.int32)
        pools.append(ids)
    # requests start with a history of held blocks so the windows free some
    rows, used = [], [0, 0]
    for _ in range(R):
        comp = int(rng.integers(0, 300))
        blocks = []
        for g, (bs, _, _) in enumerate(groups):
            k = -(-comp // bs)
            blocks.append(pools[g][used[g]:used[g] + k])
            used[g] += k
        toks = rng.integers(0, 1000, comp + 1)
        r1 = st.add_request(toks, comp, blocks)
        r2 = orc.add_request(toks, comp, blocks)
        assert r1 == r2
        rows.append(r1)
    for g in range(2):
        free = pools[g][used[g]:used[g] + int(rng.integers(2000, 6000))]
        st.pool_reset(g, free)
        orc.pool_reset(g, free)
    for rnd in range(6):
        order = rng.permutation(R)[: int(rng.integers(1000, R + 1))]
        rr = np.array(rows, np.int32)[order]
        new = np.zeros(rr.size, np.int32)
        la = np.zeros(rr.size, np.int32)
        for k, r in enumerate(rr):
            room = L - st.row_info(int(r))["completed"] - 3
            new[k] = int(rng.integers(0, max(1, min(room, 40))))
            la[k] = int(rng.integers(0, 3))
        got = st.allocate_slots(rr, new, la, windows, wm)
        want = orc.allocate_slots(rr, new, la, windows, wm)
        assert got[0] == want[0], rnd
        np.testing.assert_array_equal(got[1], want[1])
        for r, k in zip(rr[:got[0]], new[:got[0]]):
            c = st.row_info(int(r))["completed"]
            nt = st.row_info(int(r))["n_tokens"]
            extra = max(0, c + int(k) - nt)
            toks = rng.integers(0, 1000, extra)
            st.update_request(int(r), None, toks, c + int(k))
            orc.update_request(int(r), None, toks, c + int(k))
        _same_state(st, orc, R, 2)
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("R,groups,windows", [
    (16384, [(4, 24, 200000), (16, 8, 60000)], [0, 24]),                 # the largest batch
    (2000, [(bs, 20, 30000) for bs in (1, 2, 3, 4, 5, 8, 16, 32)],       # eight groups
     [0, 5, 0, 9, 0, 33, 0, 64]),
])
def test_allocate_largest_batch_and_eight_groups(R, groups, windows):
    """allocate_slots at PKV_MAX_BATCH requests (16 per thread of the
    one-CTA plan kernel) and with eight KV-cache groups, against the oracle:
    admission, new-block counts, tables and stacks."""
    rng = np.random.default_rng(R + len(groups))
    L = min(W * bs for bs, W, _ in groups) - 8
    st = pkv.State(R, L, groups)
    orc = oracle.OracleState(R, L, groups)
    pools, used, rows = [], [0] * len(groups), []
    for g, (_, _, nbk) in enumerate(groups):
        pools.append(rng.permutation(nbk).astype(np.int32))
    for _ in range(R):
        comp = int(rng.integers(0, L // 2))
        blocks = []
        for g, (bs, _, _) in enumerate(groups):
            k = -(-comp // bs)
            blocks.append(pools[g][used[g]:used[g] + k])
            used[g] += k
        toks = rng.integers(0, 1000, comp + 1)
        r1 = st.add_request(toks, comp, blocks)
        r2 = orc.add_request(toks, comp, blocks)
        assert r1 == r2
        rows.append(r1)
    for g in range(len(groups)):
        free = pools[g][used[g]:]
        free = free[: int(len(free) * 0.7)]
        st.pool_reset(g, free)
        orc.pool_reset(g, free)
    rr = np.array(rows, np.int32)[rng.permutation(R)]
    new = np.array([int(rng.integers(0, max(1, min(L - st.row_info(int(r))["completed"] - 3, 6))))
                    for r in rr], np.int32)
    la = rng.integers(0, 2, R).astype(np.int32)
    got = st.allocate_slots(rr, new, la, windows, 1)
    want = orc.allocate_slots(rr, new, la, windows, 1)
    assert got[0] == want[0]
    np.testing.assert_array_equal(got[1], want[1])
    for g in range(len(groups)):
        assert st.pool_size(g) == len(orc.pool(g)), g
        np.testing.assert_array_equal(st.pool(g), orc.pool(g))
    # every row's tables (a sample of rows for the largest batch)
    check = rows if R <= 2000 else list(rng.choice(rows, 600, replace=False))
    for r in check:
        a = orc.read_row(int(r))
        b = st.read_row(int(r), n_tokens=0)
        for g in range(len(groups)):
            assert b["block_table"][g].tolist() == a["block_table"][g].tolist(), (r, g)
    assert st.get_error() == 0
    st.close()


def test_pool_reset_and_release_over_several_ring_pieces():
    """With a 64 KiB staging ring (16 KiB pieces), a pool of 20000 ids is
    staged in five pieces and the block moves of releasing 600 requests in
    three launches; the pools end as the oracle's."""
    rng = np.random.default_rng(77)
    R, L = 640, 256
    groups = [(16, 16, 20000), (8, 32, 12000)]
    st = pkv.State(R, L, groups, ring_bytes=64 << 10)
    orc = oracle.OracleState(R, L, groups)
    for g, (_, _, nbk) in enumerate(groups):
        ids = rng.permutation(nbk).astype(np.int32)
        st.pool_reset(g, ids)
        orc.pool_reset(g, ids)
        np.testing.assert_array_equal(st.pool(g), ids)
    # 600 requests holding blocks taken from the pools' tops (as the oracle
    # hands them out), then all released in one call
    rows = []
    for _ in range(600):
        nt = int(rng.integers(1, L))
        toks = rng.integers(0, 1000, nt)
        r1 = st.add_request(toks, 0, [[], []])
        r2 = orc.add_request(toks, 0, [[], []])
        assert r1 == r2
        rows.append(r1)
    for i0 in range(0, 600, 200):   # admission in batches the small ring can stage
        batch = rows[i0:i0 + 200]
        need = [len(orc.read_row(r)["tokens"]) for r in batch]
        got = st.allocate_slots(batch, need)
        want = orc.allocate_slots(batch, need)
        assert got[0] == want[0] == len(batch)
        np.testing.assert_array_equal(got[1], want[1])
    _same_state(st, orc, R, 2)
    st.release_blocks(rows)
    orc.release_blocks(rows)
    _same_state(st, orc, R, 2)
    st.close()
