"""Helpers for the GPU parity tests: build the CUDA library's state and the
oracle's state from the same workload, and compare a prepared batch element
by element."""
from __future__ import annotations

import numpy as np

import oracle
import paged_kv_prep_gb300 as pkv
from tests.helpers import apply_ops, group_tuples, schedule_arrays


def build_states(wl, ring_bytes=0):
    st = pkv.State(wl.max_reqs, wl.max_model_len, group_tuples(wl), ring_bytes=ring_bytes)
    orc = oracle.OracleState(wl.max_reqs, wl.max_model_len, group_tuples(wl))
    rows_lib = apply_ops(st, wl)
    rows_orc = apply_ops(orc, wl)
    assert rows_lib == rows_orc, "row assignment differs from the oracle"
    return st, orc, rows_lib


def to_np(t):
    return t.detach().cpu().numpy()


def compare_batch(batch, ref, groups):
    """Every output of the GPU batch equals the oracle's, bit for bit."""
    n = len(ref["index_mapping"])
    T = ref["total_tokens"]
    assert batch.total_tokens == T
    np.testing.assert_array_equal(to_np(batch.index_mapping)[:n], ref["index_mapping"])
    np.testing.assert_array_equal(to_np(batch.query_start_loc)[:n + 1], ref["query_start_loc"])
    np.testing.assert_array_equal(to_np(batch.seq_lens)[:n], ref["seq_lens"])
    np.testing.assert_array_equal(to_np(batch.positions)[:T], ref["positions"])
    np.testing.assert_array_equal(to_np(batch.input_ids)[:T], ref["input_ids"])
    for g in range(groups):
        np.testing.assert_array_equal(to_np(batch.block_tables[g])[:n], ref["block_tables"][g])
        np.testing.assert_array_equal(to_np(batch.slot_mapping[g])[:T], ref["slot_mapping"][g])


def prepare_both(st, orc, wl, rows_map, flags=0):
    rows, ns = schedule_arrays(wl, rows_map)
    batch = st.prepare_batch(rows, ns, flags=flags)
    ref = orc.prepare_batch(rows, ns, advance=bool(flags & pkv.ADVANCE))
    return batch, ref, rows, ns
