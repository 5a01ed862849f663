"""Helpers shared by the tests: applying a workload's add/remove program to a
state (the oracle's or the CUDA library's; both expose add_request and
remove_request), and building the schedule arrays."""
from __future__ import annotations

import numpy as np


def apply_ops(state, wl):
    """Apply ``wl.ops`` in order; return {handle: row}."""
    rows = {}
    for op in wl.ops:
        if op[0] == "add":
            r = op[1]
            rows[r.handle] = state.add_request(r.token_ids, r.num_computed, r.blocks)
        else:
            state.remove_request(rows.pop(op[1]))
    return rows


def schedule_arrays(wl, rowmap):
    rows = np.array([rowmap[h] for h, _ in wl.schedule], dtype=np.int32)
    ns = np.array([c for _, c in wl.schedule], dtype=np.int32)
    return rows, ns


def group_tuples(wl):
    return [(g.block_size, g.max_blocks_per_req, g.num_blocks) for g in wl.groups]
