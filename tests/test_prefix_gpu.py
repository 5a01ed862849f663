"""Prefix-cache keys and matching on the GPU against the CPU oracle."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def _u64(t):
    return t.cpu().numpy().view(np.uint64)


def _shared_prefix_requests(rng, num, prompts, max_suffix, max_prompt):
    """Requests whose tokens are one of a few shared prompts plus a suffix."""
    bank = [rng.integers(0, 128000, int(rng.integers(0, max_prompt + 1))).astype(np.int32)
            for _ in range(prompts)]
    out = []
    for _ in range(num):
        p = bank[int(rng.integers(0, prompts))]
        suf = rng.integers(0, 128000, int(rng.integers(0, max_suffix + 1))).astype(np.int32)
        out.append(np.concatenate([p, suf]))
    return out


@pytest.mark.parametrize("bs", [1, 3, 16, 32, 64])
def test_block_keys_match_oracle(bs):
    rng = np.random.default_rng(bs)
    reqs = _shared_prefix_requests(rng, 60, 4, 300, 2000)
    reqs.append(rng.integers(0, 128000, 3000).astype(np.int32))   # > 256 blocks at small bs
    # at bs 1: 16 digests per thread of a CTA chain exactly, one more, and
    # runs of 36 (chained in pieces)
    for n in (4096, 4097, 9000):
        reqs.append(rng.integers(0, 128000, n).astype(np.int32))
    max_len = max(len(r) for r in reqs) + 1
    st = pkv.State(len(reqs) + 4, max_len, [(16, 8, 100)])
    orc = oracle.OracleState(len(reqs) + 4, max_len, [(16, 8, 100)])
    rows = [st.add_request(r, 0, [[]]) for r in reqs]
    for r in reqs:
        orc.add_request(r, 0, [[]])
    off, keys = st.block_keys(rows, bs)
    got = _u64(keys)
    for i, (row, toks) in enumerate(zip(rows, reqs)):
        want = oracle.block_keys(toks, bs)
        assert off[i + 1] - off[i] == len(toks) // bs
        np.testing.assert_array_equal(got[off[i]:off[i + 1]], want)
    st.close()


def test_prefix_cache_example_on_gpu():
    g = json.load(open(os.path.join(HERE, "golden", "prefix_cache_example.json")))
    bs = g["block_size"]
    fx = g["fixture_choices"]
    A = fx["system_prompt"] + fx["A_suffix"]
    B = fx["system_prompt"] + fx["B_suffix"]
    P = fx["system_prompt"]
    st = pkv.State(4, 16, [(bs, 4, 100)])
    ra, rb, rp = (st.add_request(t, 0, [[]]) for t in (A, B, P))
    off, keys = st.block_keys([ra, rb, rp], bs)
    pc = pkv.PrefixCache(64)
    # A ran first: its two full prompt blocks are cached as P1, P2
    pc.insert(keys[off[0]:off[0] + 2].contiguous(),
              torch.tensor([fx["P1"], fx["P2"]], dtype=torch.int32, device="cuda"))
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    caps = torch.tensor([(len(t) - 1) // bs for t in (A, B, P)], dtype=torch.int32, device="cuda")
    hits, ids = pc.match(keys, d_off, caps)
    hits = hits.cpu().tolist()
    ids = ids.cpu().numpy()
    pr = g["printed_on_the_pages"]
    assert hits[1] * bs == pr["B_reused_tokens"]
    assert ids[off[1]:off[1] + hits[1]].tolist() == [fx[n] for n in pr["B_reused_blocks"]]
    assert hits[2] == g["derived_from_the_definitions"]["prompt_only_hit_blocks"]
    assert hits[0] == 2   # A's own prompt blocks
    pc.close()
    st.close()


@pytest.mark.parametrize("seed", [0, 1])
def test_prefix_match_matches_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    bs = 16
    reqs = _shared_prefix_requests(rng, 200, 6, 200, 1500)
    max_len = max(len(r) for r in reqs) + 1
    st = pkv.State(len(reqs), max_len, [(bs, 8, 100)])
    rows = [st.add_request(r, 0, [[]]) for r in reqs]
    off, keys = st.block_keys(rows, bs)
    k_all = _u64(keys)
    # cache the first few requests' blocks (as if they had run), in two calls
    index = {}
    ins_k, ins_v = [], []
    for i in range(12):
        for j, k in enumerate(k_all[off[i]:off[i + 1]]):
            if int(k) not in index:
                index[int(k)] = 1000 * i + j
            ins_k.append(int(k))
            ins_v.append(index[int(k)])
    pc = pkv.PrefixCache(1 << 16)
    half = len(ins_k) // 2
    for a, b in ((0, half), (half, len(ins_k))):
        kk = torch.tensor(np.array(ins_k[a:b], np.uint64).view(np.int64), device="cuda")
        vv = torch.tensor(ins_v[a:b], dtype=torch.int32, device="cuda")
        pc.insert(kk, vv)
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    caps = np.array([max(0, (len(t) - 1) // bs) for t in reqs], np.int32)
    hits, ids = pc.match(keys, d_off, torch.tensor(caps, device="cuda"))
    hits = hits.cpu().numpy()
    ids = ids.cpu().numpy()
    for i, toks in enumerate(reqs):
        want_k, want_ids = oracle.prefix_hits(k_all[off[i]:off[i + 1]], len(toks), bs, index)
        assert hits[i] == want_k, i
        seg = ids[off[i]:off[i + 1]]
        assert seg[:want_k].tolist() == want_ids.tolist(), i
        assert (seg[want_k:] == -1).all(), i
    assert (hits > 0).sum() > 50   # the shared prompts do hit
    pc.close()
    st.close()


def test_block_keys_large_step_sampled():
    """Keys of every full 32-token block of the large step's 4096 requests
    (1.4 M blocks, 939 requests on the CTA-per-request chain), computed in one
    call as the benchmark does; the 40 longest requests and 60 random ones
    are compared with the oracle's keys of the same requests' token ids, taken
    from the workload (not from the device)."""
    import pkv_workloads as workloads
    wl = workloads.large_step(seed=0, num_layers=1, pool=28610)
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows = workloads.apply_ops(st, wl)
    bs = wl.groups[0].block_size
    handles = list(rows)
    off, keys = st.block_keys([rows[h] for h in handles], bs)
    got = _u64(keys)
    reqs = wl.requests()
    lengths = np.array([len(reqs[h].token_ids) for h in handles])
    rng = np.random.default_rng(9)
    pick = set(np.argsort(-lengths)[:40].tolist()) | set(rng.choice(len(handles), 60, replace=False).tolist())
    assert int(lengths.max()) // bs > 256          # the CTA-per-request chain is covered
    for i in sorted(pick):
        toks = np.asarray(reqs[handles[i]].token_ids, np.int32)
        want = oracle.block_keys(toks, bs)
        assert off[i + 1] - off[i] == len(toks) // bs
        np.testing.assert_array_equal(got[off[i]:off[i + 1]], want)
    assert st.get_error() == 0
    st.close()


@pytest.mark.parametrize("n", [3000, 20000])
def test_match_any_batch_size_with_gaps(n):
    """Keys given directly (no state): requests of 0..40 keys, an index holding
    a random half of the keys (so later blocks are often cached past an
    uncached one), a few zero keys, caps from -1 to past the end.  3000
    requests take the flat match; 20000 (more than PKV_MAX_BATCH) the
    CTA-per-request one.  Hits and ids against the oracle."""
    rng = np.random.default_rng(7 + n)
    nk = rng.integers(0, 41, n)
    off = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
    total = int(off[-1])
    keys = rng.integers(1, 2**63, total, dtype=np.int64).astype(np.uint64)
    keys[rng.random(total) < 0.01] = 0
    cached = (rng.random(total) < 0.5) & (keys != 0)
    index = {int(k): int(v) for k, v in zip(keys[cached], np.nonzero(cached)[0])}
    caps = (rng.integers(-1, 43, n)).astype(np.int32)
    pc = pkv.PrefixCache(1 << 22)
    pc.insert(torch.tensor(keys[cached].view(np.int64), device="cuda"),
              torch.tensor(np.nonzero(cached)[0].astype(np.int32), device="cuda"))
    hits, ids = pc.match(torch.tensor(keys.view(np.int64), device="cuda"),
                         torch.tensor(off, device="cuda"), torch.tensor(caps, device="cuda"))
    hits = hits.cpu().numpy()
    ids = ids.cpu().numpy()
    for i in range(n):
        seg_keys = keys[off[i]:off[i + 1]]
        # block size 1 and n_tokens = cap + 1 make the oracle's cap this cap;
        # the oracle reads keys [0, cap), so the cap is first bounded by the
        # request's own keys, as the match bounds it
        cap = min(int(nk[i]), max(int(caps[i]), 0))
        # only the index entries of this request's own keys can match: pass
        # those (the oracle takes its index as flat arrays on every call)
        own = {int(k): index[int(k)] for k in seg_keys if int(k) in index}
        want_k, want_ids = oracle.prefix_hits(seg_keys, cap + 1, 1, own)
        assert hits[i] == want_k, i
        seg = ids[off[i]:off[i + 1]]
        assert seg[:want_k].tolist() == want_ids.tolist(), i
        assert (seg[want_k:] == -1).all(), i
    assert (hits > 0).sum() > n // 10
    pc.close()


def test_insert_keeps_first_id_and_reports_a_full_table():
    pc = pkv.PrefixCache(4)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.tensor([5, 9, 13], dtype=torch.int64, device="cuda")
    pc.insert(k, torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"), d_error=err.data_ptr())
    pc.insert(k[:1], torch.tensor([77], dtype=torch.int32, device="cuda"), d_error=err.data_ptr())
    off = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    hits, ids = pc.match(k, off, torch.tensor([3], dtype=torch.int32, device="cuda"))
    assert hits.item() == 3 and ids.cpu().tolist() == [1, 2, 3]
    assert err.item() == 0
    more = torch.tensor([17, 21, 25], dtype=torch.int64, device="cuda")
    pc.insert(more, torch.tensor([4, 5, 6], dtype=torch.int32, device="cuda"), d_error=err.data_ptr())
    assert err.item() == pkv.DEVERR_TABLE_FULL
    pc.close()
