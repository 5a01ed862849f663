"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load(path)``)
and raises AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with a planted mistake and requires that every mistake trips at least one pin.

What pins what:
  * the pages' worked example (printed values and values derived from the
    definitions) -- ``tests/golden/worked_example.json``;
  * flattening by concatenation: the batch built by Python's stable ``sorted``
    and list concatenation, a different route from the oracle's insertion sort
    and prefix-sum indexing;
  * slots by brute force: for every request, a table from position to slot
    built by enumerating (block, offset) pairs with no division or remainder;
  * invariants that follow from the definitions (unique slots, slot inside a
    block the request owns, seq_lens = completed + scheduled, ...);
  * block tables against the block lists the requests were added with;
  * the KV store against numpy's fancy-index assignment, with a sentinel-filled
    cache, negative slots, padded source strides and all 256 byte values;
  * the request-state pool: lowest-free-row reuse, resets on removal, appends;
  * the paged (CSR) block tables against the worked example and against pages
    found by walking positions one at a time;
  * FNV-1a 64 against its published test vectors
    (``tests/golden/fnv1a64_vectors.json``);
  * prefix-cache block keys against an independent Python FNV-1a with
    ``struct``'s byte layout and against the chain's closed form;
  * prefix hits against the Prefix Cache example of the scheduler page
    (``tests/golden/prefix_cache_example.json``) and the num_tokens - 1 cap;
  * allocate_slots against the same example, the watermark inequality, the
    stop at the first refusal, the free stack's order, lookahead and the
    sliding-window boundary.
"""
from __future__ import annotations

import itertools
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import pkv_workloads as workloads  # noqa: E402
from tests.helpers import apply_ops, group_tuples, schedule_arrays  # noqa: E402

GOLDEN = os.path.join(HERE, "golden", "worked_example.json")


def _state(wl, lib):
    return oracle.OracleState(wl.max_reqs, wl.max_model_len, group_tuples(wl), lib=lib)


def small_workloads():
    """Small seeded cases covering every structure of the five configurations
    plus odd block sizes (1, 3, 5) and up to eight groups (the maximum)."""
    return [
        workloads.tiny(seed=0),
        workloads.tiny(seed=1),
        workloads.decode_heavy(seed=2, num_requests=24, max_ctx=300, pool=2048),
        workloads.mixed_prefill(seed=3, budget=300, num_decode=6, chunk_lo=20,
                                chunk_hi=90, max_ctx=400, rows=48, pool=4096),
        workloads.two_groups(seed=4, num_requests=40, max_ctx=700, window=64,
                             chunk_hi=40),
        workloads.large_step(seed=5, num_requests=48, budget=200, chunk_hi=60,
                             max_ctx=2048, num_layers=1, pool=1024),
        workloads.random_small(seed=6, block_sizes=(1,), max_ctx=40, max_chunk=12),
        workloads.random_small(seed=7, block_sizes=(3, 5), num_requests=15),
        workloads.random_small(seed=8, block_sizes=(16, 4, 7), num_requests=10,
                               window=24, decode_frac=0.3),
        workloads.random_small(seed=9, block_sizes=(1, 2, 3, 4, 5, 7, 16, 64),
                               num_requests=12, max_ctx=90, window=20),   # 8 groups
    ]


# ---------------------------------------------------------------------------
def pin_worked_example(lib):
    g = json.load(open(GOLDEN))
    bs = g["block_size"]
    W = g["fixture_choices"]["max_blocks_per_req"]
    st = oracle.OracleState(16, 64, [(bs, W, 1000)], lib=lib)
    # place A on row 6 and B on row 7: fill rows 0..7, free 6 and 7, add A, B
    for _ in range(8):
        st.add_request([], 0, [[]])
    st.remove_request(6)
    st.remove_request(7)
    placed = {}
    for name in ("A", "B"):
        r = g["requests"][name]
        length = r["completed_tokens"] + dict(g["schedule_in_output_order"])[name]
        toks = [1000 * r["row"] + p for p in range(length)]
        placed[name] = st.add_request(toks, r["completed_tokens"], [r["blocks"]])
    assert placed == {"A": 6, "B": 7}, placed
    rows = [g["requests"][nm]["row"] for nm, _ in g["schedule_in_output_order"]]
    ns = [c for _, c in g["schedule_in_output_order"]]
    out = st.prepare_batch(rows, ns)
    pr = g["printed_on_the_pages"]
    assert out["query_start_loc"].tolist() == pr["query_start_loc"]
    assert out["positions"].tolist() == pr["positions"]
    ft = pr["first_token_of_B"]
    assert out["positions"][ft["flat_token_index"]] == ft["position"]
    assert out["slot_mapping"][0][ft["flat_token_index"]] == ft["slot"]
    assert out["block_tables"][0][0][ft["logic_block"]] == ft["block_table_7_1"]
    der = g["derived_from_the_definitions"]
    assert out["index_mapping"].tolist() == der["index_mapping"]
    assert out["seq_lens"].tolist() == der["seq_lens"]
    assert out["slot_mapping"][0].tolist() == der["slot_mapping"]
    fx = g["fixture_choices"]
    assert out["input_ids"].tolist() == fx["input_ids"]
    assert out["block_tables"][0].tolist() == fx["input_block_tables"]
    st.close()


def _expected_by_concatenation(wl, rowmap):
    reqs = wl.requests()
    sched = wl.schedule
    order = sorted(range(len(sched)), key=lambda i: sched[i][1])  # stable
    im, pos, ids, tok_req = [], [], [], []
    for i in order:
        h, c = sched[i]
        r = reqs[h]
        im.append(rowmap[h])
        for k in range(c):
            pos.append(r.num_computed + k)
            ids.append(int(r.token_ids[r.num_computed + k]))
            tok_req.append(h)
    counts = [sched[i][1] for i in order]
    qsl = [0] + list(itertools.accumulate(counts))
    sl = [reqs[sched[i][0]].num_computed + sched[i][1] for i in order]
    return dict(order=order, index_mapping=im, positions=pos, input_ids=ids,
                query_start_loc=qsl, seq_lens=sl, token_request=tok_req)


def pin_flatten_by_concatenation(lib):
    for wl in small_workloads():
        st = _state(wl, lib)
        rowmap = apply_ops(st, wl)
        rows, ns = schedule_arrays(wl, rowmap)
        out = st.prepare_batch(rows, ns)
        exp = _expected_by_concatenation(wl, rowmap)
        for key in ("index_mapping", "positions", "input_ids", "query_start_loc",
                    "seq_lens"):
            assert out[key].tolist() == exp[key], (wl.name, key)
        assert out["total_tokens"] == wl.total_tokens
        st.close()


def pin_slots_brute_force(lib):
    """slot of (request, position) from a table built by enumerating every
    (logical block j, offset o) pair: position j*bs+o -> block[j]*bs+o."""
    for wl in small_workloads():
        st = _state(wl, lib)
        rowmap = apply_ops(st, wl)
        rows, ns = schedule_arrays(wl, rowmap)
        out = st.prepare_batch(rows, ns)
        exp = _expected_by_concatenation(wl, rowmap)
        reqs = wl.requests()
        for g, spec in enumerate(wl.groups):
            bs = spec.block_size
            tables = {}
            for h in set(exp["token_request"]):
                table = {}
                position = 0
                for blk in reqs[h].blocks[g]:
                    for o in range(bs):
                        table[position] = int(blk) * bs + o
                        position += 1
                tables[h] = table
            want = [tables[h][p] for h, p in zip(exp["token_request"], exp["positions"])]
            assert out["slot_mapping"][g].tolist() == want, (wl.name, g)
        st.close()


def pin_invariants(lib):
    for wl in small_workloads():
        st = _state(wl, lib)
        rowmap = apply_ops(st, wl)
        rows, ns = schedule_arrays(wl, rowmap)
        out = st.prepare_batch(rows, ns)
        reqs = wl.requests()
        inv_rows = {v: k for k, v in rowmap.items()}
        qsl = out["query_start_loc"]
        n = len(ns)
        # qsl is a CSR offset array over the sorted counts
        assert qsl[0] == 0 and qsl[-1] == wl.total_tokens
        diffs = np.diff(qsl)
        assert sorted(diffs.tolist()) == sorted(ns.tolist())
        assert all(diffs[b] <= diffs[b + 1] for b in range(n - 1))
        for b in range(n):
            h = inv_rows[int(out["index_mapping"][b])]
            r = reqs[h]
            lo, hi = int(qsl[b]), int(qsl[b + 1])
            p = out["positions"][lo:hi]
            # contiguous positions starting at completed
            assert p.tolist() == list(range(r.num_computed, r.num_computed + hi - lo))
            assert out["seq_lens"][b] == r.num_computed + (hi - lo)
            assert out["input_ids"][lo:hi].tolist() == r.token_ids[p].tolist()
            for g, spec in enumerate(wl.groups):
                s = out["slot_mapping"][g][lo:hi]
                blocks = np.asarray(r.blocks[g])
                # the slot lies in the block the request's table names for pos
                assert (s // spec.block_size).tolist() == blocks[p // spec.block_size].tolist()
                assert (s % spec.block_size).tolist() == (p % spec.block_size).tolist()
        for g in range(len(wl.groups)):
            s = out["slot_mapping"][g]
            assert len(np.unique(s)) == len(s), "slots must be unique within a step"
        st.close()


def pin_block_tables(lib):
    for wl in small_workloads():
        st = _state(wl, lib)
        rowmap = apply_ops(st, wl)
        rows, ns = schedule_arrays(wl, rowmap)
        out = st.prepare_batch(rows, ns)
        reqs = wl.requests()
        inv_rows = {v: k for k, v in rowmap.items()}
        for g, spec in enumerate(wl.groups):
            bt = out["block_tables"][g]
            assert bt.shape == (len(ns), spec.max_blocks_per_req)
            for b in range(len(ns)):
                blocks = list(reqs[inv_rows[int(out["index_mapping"][b])]].blocks[g])
                want = blocks + [-1] * (spec.max_blocks_per_req - len(blocks))
                assert bt[b].tolist() == want, (wl.name, g, b)
        st.close()


def pin_kv_indices(lib):
    """Paged (CSR) block tables: the worked example's values, then for every
    small workload and group the pages found by walking positions 0 ..
    seq_len - 1 one at a time (a new page each time bs positions have
    passed; no division), and the error cases."""
    g = json.load(open(GOLDEN))
    bs = g["block_size"]
    W = g["fixture_choices"]["max_blocks_per_req"]
    st = oracle.OracleState(16, 64, [(bs, W, 1000)], lib=lib)
    for _ in range(8):
        st.add_request([], 0, [[]])
    st.remove_request(6)
    st.remove_request(7)
    for name in ("A", "B"):
        r = g["requests"][name]
        length = r["completed_tokens"] + dict(g["schedule_in_output_order"])[name]
        st.add_request([1000 * r["row"] + p for p in range(length)], r["completed_tokens"],
                       [r["blocks"]])
    rows = [g["requests"][nm]["row"] for nm, _ in g["schedule_in_output_order"]]
    ns = [c for _, c in g["schedule_in_output_order"]]
    out = st.prepare_batch(rows, ns)
    indptr, indices, last = st.kv_indices(0, out["index_mapping"], out["seq_lens"])
    want = g["paged_block_tables"]
    assert indptr.tolist() == want["kv_indptr"]
    assert indices.tolist() == want["kv_indices"]
    assert last.tolist() == want["last_page_len"]
    st.close()

    for wl in small_workloads():
        st = _state(wl, lib)
        rowmap = apply_ops(st, wl)
        rows, ns = schedule_arrays(wl, rowmap)
        out = st.prepare_batch(rows, ns)
        reqs = wl.requests()
        inv_rows = {v: k for k, v in rowmap.items()}
        n = len(ns)
        for gi, spec in enumerate(wl.groups):
            pages, lasts, starts = [], [], [0]
            for b in range(n):
                blocks = list(reqs[inv_rows[int(out["index_mapping"][b])]].blocks[gi])
                j, used = 0, 0
                for _pos in range(int(out["seq_lens"][b])):
                    if used == spec.block_size:
                        j, used = j + 1, 0
                    used += 1
                pages.extend(blocks[:j + 1])
                lasts.append(used)
                starts.append(len(pages))
            indptr, indices, last = st.kv_indices(gi, out["index_mapping"], out["seq_lens"])
            assert indptr.tolist() == starts, (wl.name, gi)
            assert indices.tolist() == pages, (wl.name, gi)
            assert last.tolist() == lasts, (wl.name, gi)
            # exactly enough room is accepted, one entry less is refused
            assert st.kv_indices(gi, out["index_mapping"], out["seq_lens"],
                                 capacity=len(pages))[0].tolist() == starts
            if pages:
                assert st.kv_indices(gi, out["index_mapping"], out["seq_lens"],
                                     capacity=len(pages) - 1, check=False) == oracle.BAD_ARG
        # a seq_len past the row's W_g pages, a zero seq_len, a free row
        spec = wl.groups[0]
        im = out["index_mapping"][:1]
        too_long = np.array([spec.max_blocks_per_req * spec.block_size + 1], np.int32)
        assert st.kv_indices(0, im, too_long, check=False) == oracle.BAD_ARG
        assert st.kv_indices(0, im, np.array([spec.max_blocks_per_req * spec.block_size],
                                             np.int32))[1].size == spec.max_blocks_per_req
        assert st.kv_indices(0, im, np.zeros(1, np.int32), check=False) == oracle.BAD_ARG
        free_rows = sorted(set(range(wl.max_reqs)) - set(rowmap.values()))
        if free_rows:
            assert st.kv_indices(0, np.array(free_rows[:1], np.int32), np.ones(1, np.int32),
                                 check=False) == oracle.BAD_ARG
        st.close()


def pin_advance(lib):
    wl = workloads.random_small(seed=11, num_requests=9, max_ctx=120, max_chunk=20)
    st = _state(wl, lib)
    rowmap = apply_ops(st, wl)
    reqs = wl.requests()
    rows, ns = schedule_arrays(wl, rowmap)
    # give every request more tokens and blocks so it can run twice
    for h, c in wl.schedule:
        r = reqs[h]
        extra_tok = np.arange(c, dtype=np.int32) + 7
        need = []
        for spec, blk in zip(wl.groups, r.blocks):
            have_pos = len(blk) * spec.block_size
            end = len(r.token_ids) + c
            k = max(0, -(-(end - have_pos) // spec.block_size))
            need.append(np.arange(k, dtype=np.int32))  # block ids 0..k-1 exist
        st.update_request(rowmap[h], need, extra_tok)
    first = st.prepare_batch(rows, ns, advance=True)
    second = st.prepare_batch(rows, ns, advance=False)
    assert (second["seq_lens"] == first["seq_lens"] + np.diff(first["query_start_loc"])).all()
    assert (second["positions"] == first["positions"] + np.repeat(
        np.diff(first["query_start_loc"]), np.diff(first["query_start_loc"]))).all()
    for h, c in wl.schedule:
        assert st.read_row(rowmap[h])["completed"] == reqs[h].num_computed + c
    st.close()


def pin_state_pool(lib):
    st = oracle.OracleState(6, 32, [(4, 5, 100), (2, 9, 50)], lib=lib)
    rows = [st.add_request([1, 2, 3], 1, [[10], [20, 21]]) for _ in range(6)]
    assert rows == [0, 1, 2, 3, 4, 5], rows
    assert st.add_request([1], 0, [[], []], check=False) == -oracle.FULL
    st.remove_request(4)
    st.remove_request(1)
    assert st.remove_request(1, check=False) == oracle.NOT_ACTIVE
    # a freed row comes back reset, and the lowest free row is reused first
    r = st.read_row(1)
    assert not r["active"] and r["completed"] == 0
    assert r["block_table"][0].tolist() == [-1] * 5
    assert r["block_table"][1].tolist() == [-1] * 9
    assert st.add_request([5, 6], 2, [[], [33]]) == 1
    assert st.add_request([], 0, [[7, 8, 9], []]) == 4
    r = st.read_row(4)
    assert r["block_table"][0].tolist() == [7, 8, 9, -1, -1]
    assert r["block_table"][1].tolist() == [-1] * 9
    r = st.read_row(1)
    assert r["tokens"].tolist() == [5, 6] and r["completed"] == 2
    # update appends blocks and tokens after what is there
    st.update_request(1, [[11, 12], [34]], [9, 9, 9], num_computed=3)
    r = st.read_row(1)
    assert r["block_table"][0].tolist() == [11, 12, -1, -1, -1]
    assert r["block_table"][1].tolist() == [33, 34] + [-1] * 7
    assert r["tokens"].tolist() == [5, 6, 9, 9, 9] and r["completed"] == 3
    assert r["num_blocks"].tolist() == [2, 2]
    # error cases: inactive row, overflowing the table, bad block id
    st.remove_request(2)
    assert st.update_request(2, [[1], []], [], check=False) == oracle.NOT_ACTIVE
    assert st.update_request(1, [[1, 2, 3, 4], []], [], check=False) == oracle.CAPACITY
    assert st.update_request(1, [[100], []], [], check=False) == oracle.BAD_ARG
    assert st.add_request([1], 0, [[0], [50]], check=False) == -oracle.BAD_ARG
    st.close()


def pin_prepare_errors(lib):
    st = oracle.OracleState(4, 16, [(4, 3, 100)], lib=lib)
    a = st.add_request(list(range(6)), 4, [[1, 2]])     # positions 4,5 in block 1
    b = st.add_request(list(range(9)), 8, [[3, 4]])     # position 8 needs block 2
    assert st.prepare_batch([a], [2], check=False) is not None
    assert st.prepare_batch([a], [3], check=False) == oracle.CAPACITY   # no token 6
    assert st.prepare_batch([b], [1], check=False) == oracle.CAPACITY   # no block 2
    assert st.prepare_batch([a, a], [1, 1], check=False) == oracle.BAD_ARG
    assert st.prepare_batch([a], [0], check=False) == oracle.BAD_ARG
    assert st.prepare_batch([3], [1], check=False) == oracle.NOT_ACTIVE
    c = st.add_request(list(range(10)), 8, [[-1, 5, 6]])  # freed block 0
    out = st.prepare_batch([c], [2])
    assert out["slot_mapping"][0].tolist() == [6 * 4 + 0, 6 * 4 + 1]
    d = st.add_request(list(range(10)), 2, [[-1, 5, 6]])  # needs the freed block
    assert st.prepare_batch([d], [1], check=False) == oracle.CAPACITY
    empty = st.prepare_batch([], [])
    assert empty["query_start_loc"].tolist() == [0] and empty["total_tokens"] == 0
    st.close()


def pin_kv_write(lib):
    rng = np.random.default_rng(21)
    for line, T, num_slots, pad in ((32, 7, 40, 0), (48, 33, 64, 16), (256, 5, 9, 0)):
        src_k = rng.integers(0, 256, size=(T, line + pad), dtype=np.uint8)
        src_v = rng.integers(0, 256, size=(T, line + pad), dtype=np.uint8)
        k = src_k[:, :line]
        v = src_v[:, :line]
        slots = rng.permutation(num_slots)[:T].astype(np.int64)
        slots[rng.uniform(size=T) < 0.2] = -1
        kc = np.full((num_slots, line), 0xA5, np.uint8)
        vc = np.full((num_slots, line), 0x5A, np.uint8)
        assert oracle.kv_write(k, v, kc, vc, slots, lib=lib) == oracle.OK
        ek = np.full((num_slots, line), 0xA5, np.uint8)
        ev = np.full((num_slots, line), 0x5A, np.uint8)
        keep = slots >= 0
        ek[slots[keep]] = k[keep]
        ev[slots[keep]] = v[keep]
        assert (kc == ek).all() and (vc == ev).all()
    # every byte value survives (fp8 bit patterns, NaNs included)
    T, line = 4, 256
    k = np.tile(np.arange(256, dtype=np.uint8), (T, 1))
    v = k[:, ::-1].copy()
    kc = np.zeros((8, line), np.uint8)
    vc = np.zeros((8, line), np.uint8)
    slots = np.array([5, 0, 7, 2], np.int64)
    assert oracle.kv_write(k, v, kc, vc, slots, lib=lib) == oracle.OK
    assert (kc[slots] == k).all() and (vc[slots] == v).all()
    # a slot past the cache is refused and nothing is written
    kc2 = kc.copy()
    assert oracle.kv_write(k, v, kc2, vc.copy(), np.array([1, 2, 3, 8], np.int64),
                           lib=lib) == oracle.BAD_ARG
    assert (kc2 == kc).all()


def pin_fnv_vectors(lib):
    g = json.load(open(os.path.join(HERE, "golden", "fnv1a64_vectors.json")))
    for v in g["vectors"]:
        assert oracle.fnv1a64(v["input"].encode(), lib=lib) == int(v["fnv1a64"], 16), v


def pin_prefix_cache_example(lib):
    g = json.load(open(os.path.join(HERE, "golden", "prefix_cache_example.json")))
    bs = g["block_size"]
    fx = g["fixture_choices"]
    A = fx["system_prompt"] + fx["A_suffix"]
    B = fx["system_prompt"] + fx["B_suffix"]
    ka = oracle.block_keys(A, bs, lib=lib)
    kb = oracle.block_keys(B, bs, lib=lib)
    # A ran first: its two full prompt blocks are cached as P1, P2
    index = {int(ka[0]): fx["P1"], int(ka[1]): fx["P2"]}
    hits, ids = oracle.prefix_hits(kb, len(B), bs, index, lib=lib)
    pr = g["printed_on_the_pages"]
    assert hits * bs == pr["B_reused_tokens"]
    assert ids.tolist() == [fx[name] for name in pr["B_reused_blocks"]]
    assert len(B) - hits * bs == pr["B_suffix_tokens"]
    # B's table: the reused blocks, then one newly allocated block for the suffix
    table = ids.tolist() + [fx["B3"]] * (-(-(len(B) - hits * bs) // bs))
    assert table == [fx[name] for name in pr["B_logical_block_table"]]
    der = g["derived_from_the_definitions"]
    assert hits == der["B_hit_blocks"]
    prompt = fx["system_prompt"]
    hp, _ = oracle.prefix_hits(oracle.block_keys(prompt, bs, lib=lib), len(prompt), bs, index,
                               lib=lib)
    assert hp == der["prompt_only_hit_blocks"]


def _fnv_py(data):
    h = 0xcbf29ce484222325
    for b in data:
        h = ((h ^ b) * 0x100000001b3) % (1 << 64)
    return h


def pin_block_keys(lib):
    """Keys by a different route: Python's struct for the byte layout, a
    Python FNV-1a (checked on the published vectors first) and the closed
    form key_j = P^(j+1) * basis + sum_i P^(j-i) * digest_i (mod 2^64)."""
    import struct
    g = json.load(open(os.path.join(HERE, "golden", "fnv1a64_vectors.json")))
    for v in g["vectors"]:
        assert _fnv_py(v["input"].encode()) == int(v["fnv1a64"], 16)
    P, basis, M = 0x100000001b3, 0xcbf29ce484222325, 1 << 64
    rng = np.random.default_rng(77)
    for bs in (1, 3, 16, 32):
        tok = rng.integers(-2**31, 2**31, size=int(rng.integers(0, 200)), dtype=np.int64)
        tok = tok.astype(np.int32)
        keys = oracle.block_keys(tok, bs, lib=lib)
        nfull = len(tok) // bs
        assert len(keys) == nfull
        digests = [_fnv_py(struct.pack("<%di" % bs, *tok[j * bs:(j + 1) * bs].tolist()))
                   for j in range(nfull)]
        for j in range(nfull):
            want = pow(P, j + 1, M) * basis
            for i in range(j + 1):
                want += pow(P, j - i, M) * digests[i]
            assert int(keys[j]) == want % M, (bs, j)
        # a key depends on its block and everything before it, nothing after
        if nfull >= 3:
            assert oracle.block_keys(tok[: 2 * bs], bs, lib=lib).tolist() == keys[:2].tolist()
            swapped = tok.copy()
            swapped[:bs], swapped[bs:2 * bs] = tok[bs:2 * bs].copy(), tok[:bs].copy()
            ks = oracle.block_keys(swapped, bs, lib=lib)
            if not np.array_equal(tok[:bs], tok[bs:2 * bs]):
                assert ks[1] != keys[1] and ks[2] != keys[2]
    # same block content after different prefixes: different keys
    a = oracle.block_keys([1, 2, 3, 4, 9, 9, 9, 9], 4, lib=lib)
    b = oracle.block_keys([5, 6, 7, 8, 9, 9, 9, 9], 4, lib=lib)
    assert a[1] != b[1]


def pin_prefix_hits(lib):
    rng = np.random.default_rng(78)
    bs = 4
    base = rng.integers(0, 1000, 40).astype(np.int32)
    keys = oracle.block_keys(base, bs, lib=lib)
    index = {int(k): 100 + j for j, k in enumerate(keys[:6])}
    # hits stop at the first uncached block and at floor((n - 1) / bs)
    for n in range(0, 41):
        hits, ids = oracle.prefix_hits(keys[: n // bs], n, bs, index, lib=lib)
        want = min(6, max(0, (n - 1) // bs)) if n > 0 else 0
        assert hits == want, (n, hits)
        assert ids.tolist() == [100 + j for j in range(want)]
    gap = dict(index)
    del gap[int(keys[2])]
    assert oracle.prefix_hits(keys, 40, bs, gap, lib=lib)[0] == 2


def pin_allocate_slots(lib):
    g = json.load(open(os.path.join(HERE, "golden", "prefix_cache_example.json")))
    bs = g["block_size"]
    fx = g["fixture_choices"]
    B = fx["system_prompt"] + fx["B_suffix"]
    st = oracle.OracleState(8, 64, [(bs, 8, 100)], lib=lib)
    st.pool_reset(0, [70, 71, fx["B3"]])          # B3 on top of the free stack
    # B arrives with its prefix hit attached (P1, P2: 8 tokens computed)
    rb = st.add_request(B, 8, [[fx["P1"], fx["P2"]]])
    adm, nb = st.allocate_slots([rb], [len(B) - 8])
    pr = g["printed_on_the_pages"]
    assert adm == 1 and nb.tolist() == [[len(pr["B_newly_allocated"])]]
    table = st.read_row(rb)["block_table"][0]
    assert table[:3].tolist() == [fx[name] for name in pr["B_logical_block_table"]]
    assert st.pool(0).tolist() == [70, 71]
    # admission: available = free - 0 reserved; required = new + watermark
    st2 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st2.pool_reset(0, list(range(5)))
    a = st2.add_request(list(range(40)), 0, [[]])
    assert st2.allocate_slots([a], [12], watermark=2)[0] == 1      # 3 + 2 <= 5
    b = st2.add_request(list(range(40)), 0, [[]])
    assert st2.allocate_slots([b], [8], watermark=1)[0] == 0       # 2 + 1 > 2
    assert st2.pool(0).tolist() == [0, 1]
    # a refused request stops the batch; later ones are not admitted
    st3 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st3.pool_reset(0, list(range(6)))
    rs = [st3.add_request(list(range(40)), 0, [[]]) for _ in range(3)]
    adm, nb = st3.allocate_slots(rs, [4, 24, 1])   # 1 block fits; 6 > 5 left
    assert adm == 1 and nb.tolist() == [[1], [0], [0]]
    # LIFO: ids come off the top, request after request
    st4 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st4.pool_reset(0, [10, 11, 12, 13, 14])
    r0 = st4.add_request(list(range(40)), 0, [[]])
    r1 = st4.add_request(list(range(40)), 0, [[]])
    st4.allocate_slots([r0, r1], [8, 4])
    assert st4.read_row(r0)["block_table"][0][:2].tolist() == [14, 13]
    assert st4.read_row(r1)["block_table"][0][:1].tolist() == [12]
    # speculative lookahead counts toward the slots needed: 7 + 1 + 1 = 9
    # tokens need 3 blocks of 4, one more than the 2 held
    st6 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st6.pool_reset(0, [5, 6])
    r6 = st6.add_request(list(range(9)), 7, [[1, 2]])
    assert st6.allocate_slots([r6], [1], lookahead=[1])[1].tolist() == [[1]]
    assert st6.allocate_slots([r6], [1], lookahead=[0])[1].tolist() == [[0]]
    # sliding window 8, bs 4: at computed 20 the window starts at 13, so the
    # blocks wholly before it (0, 1, 2) are freed
    st5 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st5.pool_reset(0, [90])
    r = st5.add_request(list(range(22)), 20, [[40, 41, 42, 43, 44, 45]])
    adm, nb = st5.allocate_slots([r], [2], windows=[8])
    assert adm == 1 and nb.tolist() == [[0]]
    assert st5.read_row(r)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, 45]
    assert st5.pool(0).tolist() == [90, 40, 41, 42]
    # at computed 19 the window starts at 12: blocks 0..2 are wholly before it
    st7 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st7.pool_reset(0, [])
    r7 = st7.add_request(list(range(20)), 19, [[30, 31, 32, 33, 34]])
    st7.allocate_slots([r7], [1], windows=[8])
    assert st7.read_row(r7)["block_table"][0][:5].tolist() == [-1, -1, -1, 33, 34]
    assert st7.pool(0).tolist() == [30, 31, 32]
    # the page's order: step (2) frees come before the check of step (4), so
    # they can serve the request itself.  Empty pool, computed 20, five
    # blocks, 4 new tokens: 24 slots need 6 blocks (1 missing) and blocks
    # 0..2 leave the window; with 3 free blocks 1 + 0 <= 3, so the request is
    # admitted and takes the last id pushed
    st8 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st8.pool_reset(0, [])
    r8 = st8.add_request(list(range(24)), 20, [[40, 41, 42, 43, 44]])
    adm, nb = st8.allocate_slots([r8], [4], windows=[8])
    assert adm == 1 and nb.tolist() == [[1]]
    assert st8.read_row(r8)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, 42]
    assert st8.pool(0).tolist() == [40, 41]
    # one request's frees serve the next one of the same call
    st9 = oracle.OracleState(4, 64, [(4, 8, 100)], lib=lib)
    st9.pool_reset(0, [])
    a9 = st9.add_request(list(range(22)), 20, [[40, 41, 42, 43, 44, 45]])
    b9 = st9.add_request(list(range(8)), 0, [[]])
    adm, nb = st9.allocate_slots([a9, b9], [2, 8], windows=[8])
    assert adm == 2 and nb.tolist() == [[0], [2]]
    assert st9.read_row(b9)["block_table"][0][:3].tolist() == [42, 41, -1]
    assert st9.pool(0).tolist() == [40]
    # a refused request's frees stand (step 2 precedes the check): 40 slots
    # need 10 blocks, 5 missing, 3 free
    st10 = oracle.OracleState(4, 64, [(4, 12, 100)], lib=lib)
    st10.pool_reset(0, [])
    r10 = st10.add_request(list(range(40)), 20, [[40, 41, 42, 43, 44]])
    adm, nb = st10.allocate_slots([r10], [20], windows=[8])
    assert adm == 0 and nb.tolist() == [[0]]
    assert st10.read_row(r10)["block_table"][0][:6].tolist() == [-1, -1, -1, 43, 44, -1]
    assert st10.pool(0).tolist() == [40, 41, 42]
    # a row listed twice is rejected before anything changes
    assert st10.allocate_slots([r10, r10], [1, 1], windows=[8], check=False) != 0
    assert st10.pool(0).tolist() == [40, 41, 42]
    # release: the held blocks go back, in logical order
    st5.release_blocks([r])
    assert st5.pool(0).tolist() == [90, 40, 41, 42, 43, 44, 45]
    assert st5.read_row(r)["block_table"][0][:6].tolist() == [-1] * 6


PINS = [pin_worked_example, pin_flatten_by_concatenation, pin_slots_brute_force,
        pin_invariants, pin_block_tables, pin_kv_indices, pin_advance, pin_state_pool,
        pin_prepare_errors, pin_kv_write, pin_fnv_vectors, pin_prefix_cache_example,
        pin_block_keys, pin_prefix_hits, pin_allocate_slots]


def run_all(path=None):
    """Run every pin on the oracle library at ``path``; return failing names."""
    lib = oracle.load(path)
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 -- any failure counts
            failed.append(f"{pin.__name__}: {type(e).__name__}: {e}")
    return failed


if __name__ == "__main__":
    bad = run_all(sys.argv[1] if len(sys.argv) > 1 else None)
    for b in bad:
        print(b)
    sys.exit(1 if bad else 0)
