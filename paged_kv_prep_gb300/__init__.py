"""paged_kv_prep_gb300: per-step GPU input preparation and paged-KV store for
a vLLM-style worker, written for one GB300 (sm_103a).

The compute lives in the CUDA library ``libpkv.so`` (C ABI in
``include/pkv.h``); this package is its thin Python binding.  PyTorch provides
device memory and streams only.

    state = State(max_reqs, max_model_len, [(block_size, W, num_blocks), ...])
    row = state.add_request(token_ids, num_computed, [blocks_g0, ...])
    batch = state.prepare_batch(rows, num_scheduled_tokens)
    kv_cache_write(k, v, k_cache, v_cache, batch.slot_mapping[0])
"""
from ._lib import (  # noqa: F401
    ADVANCE, LIVE_TABLES, SCHEDULE_SETTLED, DEVERR_BLOCK, DEVERR_DUP, DEVERR_OUTPUT_FULL, DEVERR_TABLE_FULL, DEVERR_TIMEOUT, DEVERR_COUNT, DEVERR_POSITION, DEVERR_ROW, DEVERR_SLOT,
    ERR_ALIGN, ERR_CAPACITY, ERR_CUDA, ERR_DEVICE, ERR_FULL, ERR_INVALID_ARG,
    ERR_NOT_ACTIVE, EXPORTS, MAX_BATCH, MAX_GROUPS, OK, Batch, KvStepCall, KvStoreCall,
    PkvError, PrefixCache, PrepareDeviceCall, PrepareHostCall, State, kv_cache_write, kv_cache_write_layers,
    kv_cache_write_step, lib, selftest_wait_timeout,
)

__version__ = "0.1.0"
