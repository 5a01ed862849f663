"""kv_cache_write on the GPU against the CPU oracle.

Small caches are compared in full (every byte) with the oracle's store on the
CPU.  At full size the written lines are compared with their source lines at
the oracle's slots, and every line that no slot names must still hold the
sentinel the cache was filled with."""
import numpy as np
import pytest

import oracle
import paged_kv_prep_gb300 as pkv
import pkv_workloads as workloads
from tests.gpu_helpers import build_states, compare_batch, prepare_both, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield
    torch.cuda.empty_cache()


def _sentinel_slice(a, b, line, salt):
    """Lines a..b of a cache filled with a pattern that differs per slot and
    per byte: (hash(slot) + 7 * byte + salt) mod 256."""
    sl = torch.arange(a, b, device="cuda", dtype=torch.int64)
    h = ((sl * 2654435761 + salt * 97) >> 13).to(torch.uint8)
    by = ((torch.arange(line, device="cuda", dtype=torch.int64) * 7 + salt) & 255).to(torch.uint8)
    return h[:, None] + by[None, :]


def _sentinel(num_slots, line, salt):
    out = torch.empty(num_slots, line, dtype=torch.uint8, device="cuda")
    step = max(1, (256 << 20) // line)
    for a in range(0, num_slots, step):
        b = min(num_slots, a + step)
        out[a:b] = _sentinel_slice(a, b, line, salt)
    return out


def _oracle_store(k, v, kc, vc, slots):
    kc_h, vc_h = to_np(kc).copy(), to_np(vc).copy()
    rc = oracle.kv_write(to_np(k), to_np(v), kc_h, vc_h, to_np(slots))
    assert rc == oracle.OK
    return kc_h, vc_h


@pytest.mark.parametrize("line,T,num_slots,pad", [
    (2048, 37, 300, 0),     # fp16/bf16 H8 x D128
    (1024, 200, 1000, 0),   # fp8 H8 x D128
    (512, 64, 100, 512),    # strided sources (K/V views of a wider buffer)
    (4096, 9, 40, 0),
    (16, 333, 500, 16),     # generic path: lines that are not a multiple of 512
    (48, 70, 80, 0),
    (1040, 50, 64, 32),
])
def test_store_matches_oracle(line, T, num_slots, pad):
    g = torch.Generator(device="cuda")
    g.manual_seed(line * 7 + T)
    wide_k = torch.randint(0, 256, (T, line + pad), generator=g, device="cuda", dtype=torch.uint8)
    wide_v = torch.randint(0, 256, (T, line + pad), generator=g, device="cuda", dtype=torch.uint8)
    k, v = wide_k[:, :line], wide_v[:, :line]
    perm = torch.randperm(num_slots, generator=g, device="cuda")[:T].to(torch.int64)
    drop = torch.rand(T, generator=g, device="cuda") < 0.15
    slots = torch.where(drop, torch.full_like(perm, -1), perm)
    kc = _sentinel(num_slots, line, 1)
    vc = _sentinel(num_slots, line, 2)
    want_k, want_v = _oracle_store(k, v, kc, vc, slots)
    pkv.kv_cache_write(k, v, kc, vc, slots)
    np.testing.assert_array_equal(to_np(kc), want_k)
    np.testing.assert_array_equal(to_np(vc), want_v)


@pytest.mark.parametrize("tp", [2, 4])
def test_head_shards_match_full_line_store(tp):
    """Tensor parallelism over KV heads: rank r holds heads [r H/tp, (r+1) H/tp)
    of every line in a cache of its own and stores them from a strided view of
    the fused K/V rows.  Each shard's cache equals the matching column block of
    the oracle's full-line store, with the same slot_mapping on every rank."""
    T, num_slots, line = 96, 400, 2048          # bf16, H = 8, D = 128
    g = torch.Generator(device="cuda")
    g.manual_seed(77 + tp)
    k = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
    v = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
    slots = torch.randperm(num_slots, generator=g, device="cuda")[:T].to(torch.int64)
    kc_full = _sentinel(num_slots, line, 3)
    vc_full = _sentinel(num_slots, line, 4)
    want_k, want_v = _oracle_store(k, v, kc_full, vc_full, slots)
    w = line // tp
    for r in range(tp):
        kc = kc_full[:, r * w:(r + 1) * w].contiguous()
        vc = vc_full[:, r * w:(r + 1) * w].contiguous()
        pkv.kv_cache_write(k[:, r * w:(r + 1) * w], v[:, r * w:(r + 1) * w], kc, vc, slots)
        np.testing.assert_array_equal(to_np(kc), want_k[:, r * w:(r + 1) * w])
        np.testing.assert_array_equal(to_np(vc), want_v[:, r * w:(r + 1) * w])


def test_every_byte_value_survives():
    """fp8 e4m3 lines holding all 256 bit patterns (NaNs included) arrive
    unchanged: the store never goes through a float conversion."""
    T, line = 64, 1024
    k = workloads.all_byte_values_source(T, line, device="cuda")
    v = workloads.all_byte_values_source(T, line, device="cuda", shift=101)
    kf8 = k.view(torch.float8_e4m3fn)
    kc = torch.zeros(128, line, dtype=torch.uint8, device="cuda")
    vc = torch.zeros(128, line, dtype=torch.uint8, device="cuda")
    slots = torch.arange(T, device="cuda", dtype=torch.int64) * 2 + 1
    pkv.kv_cache_write(kf8, v, kc.view(torch.float8_e4m3fn), vc, slots)
    assert torch.equal(kc[1::2][:T], k) and torch.equal(vc[1::2][:T], v)
    assert int(kc[0::2].sum()) == 0


def test_multi_layer_store_matches_single_layer_calls():
    L, T, line, num_slots = 130, 100, 512, 600   # more layers than one launch takes (128)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    ks = [torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
          for _ in range(L)]
    vs = [torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
          for _ in range(L)]
    slots = torch.randperm(num_slots, generator=g, device="cuda")[:T].to(torch.int64)
    a_k = [_sentinel(num_slots, line, i) for i in range(L)]
    a_v = [_sentinel(num_slots, line, 100 + i) for i in range(L)]
    b_k = [t.clone() for t in a_k]
    b_v = [t.clone() for t in a_v]
    for i in range(L):
        pkv.kv_cache_write(ks[i], vs[i], a_k[i], a_v[i], slots)
    pkv.kv_cache_write_layers(ks, vs, b_k, b_v, slots)
    for i in range(L):
        assert torch.equal(a_k[i], b_k[i]) and torch.equal(a_v[i], b_v[i])
    want_k, want_v = _oracle_store(ks[3], vs[3], _sentinel(num_slots, line, 3),
                                   _sentinel(num_slots, line, 103), slots)
    np.testing.assert_array_equal(to_np(b_k[3]), want_k)
    np.testing.assert_array_equal(to_np(b_v[3]), want_v)


def test_slot_past_cache_is_flagged_and_skipped():
    st = pkv.State(2, 8, [(4, 2, 10)])
    T, line = 4, 32
    k = torch.randint(0, 256, (T, line), device="cuda", dtype=torch.uint8)
    kc = torch.zeros(10, line, dtype=torch.uint8, device="cuda")
    vc = torch.zeros(10, line, dtype=torch.uint8, device="cuda")
    slots = torch.tensor([0, 10, -1, 9], dtype=torch.int64, device="cuda")
    pkv.kv_cache_write(k, k, kc, vc, slots, d_error=st.error_word)
    assert st.get_error() == pkv.DEVERR_SLOT
    assert torch.equal(kc[0], k[0]) and torch.equal(kc[9], k[3])
    assert int(kc[1:9].sum()) == 0
    st.close()


def test_alignment_is_checked():
    k = torch.zeros(8, 64, dtype=torch.uint8, device="cuda")
    kc = torch.zeros(16, 64, dtype=torch.uint8, device="cuda")
    slots = torch.arange(8, dtype=torch.int64, device="cuda")
    back = torch.zeros(16 * 64 + 8, dtype=torch.uint8, device="cuda")
    bad = back[8:].view(16, 64)
    assert pkv.kv_cache_write(k, k, bad, kc, slots, check=False) == pkv.ERR_ALIGN
    k2 = torch.zeros(8, 72, dtype=torch.uint8, device="cuda")[:, :64]   # 72-byte stride
    assert pkv.kv_cache_write(k2, k, kc, kc, slots, check=False) == pkv.ERR_ALIGN
    assert pkv.kv_cache_write(k, k, kc, kc, slots[:0], check=False) == pkv.OK


def _check_written_and_untouched(kc, vc, k, v, slots_t, salt_k, salt_v):
    keep = slots_t >= 0
    s = slots_t[keep]
    assert torch.equal(kc[s], k[keep]) and torch.equal(vc[s], v[keep])
    mask = torch.ones(kc.shape[0], dtype=torch.bool, device="cuda")
    mask[s] = False
    num_slots, line = kc.shape
    # untouched lines still hold the sentinel, compared in pieces
    step = max(1, (256 << 20) // line)
    for a in range(0, num_slots, step):
        b = min(num_slots, a + step)
        m = mask[a:b]
        exp_k = _sentinel_slice(a, b, line, salt_k)
        exp_v = _sentinel_slice(a, b, line, salt_v)
        assert torch.equal(kc[a:b][m], exp_k[m]) and torch.equal(vc[a:b][m], exp_v[m])


@pytest.mark.parametrize("name", ["tiny", "decode_heavy", "mixed_prefill", "two_groups"])
def test_step_store_full_size(name):
    """One step of the configuration at full size: prepare on the GPU (checked
    against the oracle), then the KV store of every group at the oracle's
    slots, with the written and untouched lines checked."""
    wl = workloads.build(name, seed=1)
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, len(wl.groups))
    line = wl.line_bytes
    for g, spec in enumerate(wl.groups):
        num_slots = spec.num_blocks * spec.block_size
        kc = _sentinel(num_slots, line, 11 + g)
        vc = _sentinel(num_slots, line, 21 + g)
        k, v = workloads.kv_sources(wl, 0, g, device="cuda", row_pad=0 if g == 0 else 256)
        pkv.kv_cache_write(k, v, kc, vc, batch.slot_mapping[g], d_error=st.error_word)
        slots_ref = torch.from_numpy(ref["slot_mapping"][g]).cuda()
        _check_written_and_untouched(kc, vc, k, v, slots_ref, 11 + g, 21 + g)
        del kc, vc
        torch.cuda.empty_cache()
    assert st.get_error() == 0
    st.close()


def test_large_step_80_layers_full_size():
    """The large step at full size in the launch configuration the benchmark
    times: 80 per-layer caches of 28,610 blocks x 32 slots x 1 KiB (fp8),
    written by one multi-layer launch; every layer's written lines and a
    sample of layers' untouched lines are checked."""
    wl = workloads.large_step(seed=0)
    st, orc, rows = build_states(wl)
    batch, ref, _, _ = prepare_both(st, orc, wl, rows)
    compare_batch(batch, ref, 1)
    spec = wl.groups[0]
    num_slots = spec.num_blocks * spec.block_size
    line = wl.line_bytes
    L = wl.num_layers
    kcs, vcs, ks, vs = [], [], [], []
    for layer in range(L):
        kcs.append(_sentinel(num_slots, line, 1000 + layer))
        vcs.append(_sentinel(num_slots, line, 2000 + layer))
        k, v = workloads.kv_sources(wl, layer, 0, device="cuda")
        ks.append(k)
        vs.append(v)
    pkv.kv_cache_write_layers(ks, vs, kcs, vcs, batch.slot_mapping[0], d_error=st.error_word)
    slots_ref = torch.from_numpy(ref["slot_mapping"][0]).cuda()
    keep = slots_ref >= 0
    for layer in range(L):
        s = slots_ref[keep]
        assert torch.equal(kcs[layer][s], ks[layer][keep]), layer
        assert torch.equal(vcs[layer][s], vs[layer][keep]), layer
    for layer in (0, 41, L - 1):
        _check_written_and_untouched(kcs[layer], vcs[layer], ks[layer], vs[layer], slots_ref,
                                     1000 + layer, 2000 + layer)
    assert st.get_error() == 0
    del kcs, vcs, ks, vs
    st.close()
    torch.cuda.empty_cache()


def test_step_store_matches_separate_calls():
    """Items with their own slot_mappings and pools (two groups x three
    layers) in one launch give the same caches as one call per item, and the
    oracle's store."""
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    T, line = 500, 1024
    pools = [3000, 1200]
    items_a, items_b = [], []
    for grp, ns in enumerate(pools):
        slots = torch.randperm(ns, generator=g, device="cuda")[:T].to(torch.int64)
        slots[::13] = -1
        for layer in range(3):
            k = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
            v = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
            kc = _sentinel(ns, line, 10 * grp + layer)
            vc = _sentinel(ns, line, 50 + 10 * grp + layer)
            items_a.append((k, v, kc, vc, slots))
            items_b.append((k, v, kc.clone(), vc.clone(), slots))
    for k, v, kc, vc, sl in items_a:
        want_k, want_v = _oracle_store(k, v, kc, vc, sl)
        pkv.kv_cache_write(k, v, kc, vc, sl)
        np.testing.assert_array_equal(to_np(kc), want_k)
        np.testing.assert_array_equal(to_np(vc), want_v)
    pkv.kv_cache_write_step(items_b)
    for (_, _, ka, va, _), (_, _, kb, vb, _) in zip(items_a, items_b):
        assert torch.equal(ka, kb) and torch.equal(va, vb)
    # prebuilt call, a second time: idempotent
    pkv.KvStepCall(items_b)()
    for (_, _, ka, va, _), (_, _, kb, vb, _) in zip(items_a, items_b):
        assert torch.equal(ka, kb) and torch.equal(va, vb)
    # an item whose slot passes its own pool is flagged and skipped
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k, v, kc, vc, sl = items_b[-1]
    bad = sl.clone()
    bad[0] = kc.shape[0]
    pkv.kv_cache_write_step([(k, v, kc, vc, bad)], d_error=err.data_ptr())
    assert int(err.item()) == pkv.DEVERR_SLOT
    keep = bad >= 0
    keep[0] = False
    assert torch.equal(kc[bad[keep]], k[keep])


def test_step_store_over_one_launch_of_items():
    """130 (layer, group) items -- more than the 128 one launch's parameter
    block holds, so the call makes two launches -- give the caches one call
    per item gives."""
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    T, line = 64, 256
    pools = [700, 300]
    items_a, items_b = [], []
    for grp, ns in enumerate(pools):
        slots = torch.randperm(ns, generator=g, device="cuda")[:T].to(torch.int64)
        slots[::7] = -1
        for layer in range(65):
            k = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
            v = torch.randint(0, 256, (T, line), generator=g, device="cuda", dtype=torch.uint8)
            kc = _sentinel(ns, line, (7 * grp + layer) % 200)
            vc = _sentinel(ns, line, (11 * grp + layer + 50) % 200)
            items_a.append((k, v, kc, vc, slots))
            items_b.append((k, v, kc.clone(), vc.clone(), slots))
    for k, v, kc, vc, sl in items_a:
        pkv.kv_cache_write(k, v, kc, vc, sl)
    pkv.kv_cache_write_step(items_b)
    for (_, _, ka, va, _), (_, _, kb, vb, _) in zip(items_a, items_b):
        assert torch.equal(ka, kb) and torch.equal(va, vb)
    k, v, kc, vc, sl = items_b[129]
    want_k, want_v = _oracle_store(k, v, _sentinel(pools[1], line, (7 + 64) % 200),
                                   _sentinel(pools[1], line, (11 + 64 + 50) % 200), sl)
    np.testing.assert_array_equal(to_np(kc), want_k)
    np.testing.assert_array_equal(to_np(vc), want_v)
