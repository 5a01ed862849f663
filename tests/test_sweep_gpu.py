"""A seeded sweep of random small steps (block sizes 1 to 64, one to three
KV-cache groups, sliding windows, decode/prefill mixes, recycled rows): for
every seed the CUDA path -- host-schedule and device-schedule prepare, live
tables, the paged table of every group and the KV store -- against the oracle,
element by element."""
import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests.gpu_helpers import build_states, compare_batch, to_np
from tests.helpers import schedule_arrays

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SEEDS = list(range(100, 160))
LINE = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def random_step(seed):
    rng = np.random.default_rng([seed, 77])
    G = int(rng.integers(1, 4))
    bss = tuple(int(x) for x in rng.choice([1, 2, 3, 4, 5, 7, 8, 16, 32, 64], G))
    window = int(rng.integers(4, 200)) if rng.uniform() < 0.3 else 0
    return workloads.random_small(
        seed=seed, block_sizes=bss, num_requests=int(rng.integers(1, 121)),
        max_ctx=int(rng.integers(8, 3000)), max_chunk=int(rng.integers(1, 300)),
        decode_frac=float(rng.uniform()), window=window)


@pytest.mark.parametrize("seed", SEEDS)
def test_random_step_matches_oracle(seed):
    wl = random_step(seed)
    st, orc, rows = build_states(wl)
    r, ns = schedule_arrays(wl, rows)
    ref = orc.prepare_batch(r, ns)
    T = int(ns.sum())
    # host and device schedule paths, full tables
    compare_batch(st.prepare_batch(r, ns), ref, len(wl.groups))
    d_r = torch.tensor(r, dtype=torch.int32, device="cuda")
    d_n = torch.tensor(ns, dtype=torch.int32, device="cuda")
    batch = st.prepare_batch_device(d_r, d_n, T)
    compare_batch(batch, ref, len(wl.groups))
    # live tables: the entries attention reads
    live = st.prepare_batch(r, ns, flags=pkv.LIVE_TABLES)
    for g, spec in enumerate(wl.groups):
        got = to_np(live.block_tables[g])
        for b, sl in enumerate(ref["seq_lens"]):
            k = min(-(-int(sl) // spec.block_size), spec.max_blocks_per_req)
            np.testing.assert_array_equal(got[b, :k], ref["block_tables"][g][b, :k])
    # the paged table of every group
    for g in range(len(wl.groups)):
        w_ptr, w_idx, w_last = orc.kv_indices(g, ref["index_mapping"], ref["seq_lens"])
        indptr, indices, last = st.kv_indices(g, batch.index_mapping, batch.seq_lens)
        np.testing.assert_array_equal(to_np(indptr), w_ptr)
        np.testing.assert_array_equal(to_np(indices)[:w_ptr[-1]], w_idx)
        np.testing.assert_array_equal(to_np(last)[:len(w_last)], w_last)
    # the KV store of group 0 (64-byte lines), the whole cache compared
    spec = wl.groups[0]
    num_slots = spec.num_blocks * spec.block_size
    rng = np.random.default_rng([seed, 78])
    k = rng.integers(0, 256, (max(T, 1), LINE), dtype=np.uint8)
    v = rng.integers(0, 256, (max(T, 1), LINE), dtype=np.uint8)
    kc = np.zeros((num_slots, LINE), np.uint8)
    vc = np.zeros((num_slots, LINE), np.uint8)
    assert oracle.kv_write(k[:T], v[:T], kc, vc, ref["slot_mapping"][0]) == oracle.OK
    d_kc = torch.zeros(num_slots, LINE, dtype=torch.uint8, device="cuda")
    d_vc = torch.zeros_like(d_kc)
    pkv.kv_cache_write(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), d_kc, d_vc,
                       batch.slot_mapping[0], num_tokens=T, d_error=st.error_word)
    np.testing.assert_array_equal(to_np(d_kc), kc)
    np.testing.assert_array_equal(to_np(d_vc), vc)
    assert st.get_error() == 0
    st.close()
    orc.close()
