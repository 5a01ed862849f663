"""ctypes binding of the C ABI declared in ``include/pkv.h``.

Argument marshalling only: host arrays become int32 numpy buffers, device
buffers are torch tensors passed by pointer, streams are torch streams.  Every
step of the path runs in the CUDA library; there is no Python or CPU fallback.
If ``libpkv.so`` has not been built, every entry point raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libpkv.so")

MAX_GROUPS = 8
MAX_BATCH = 16384
STATIC_MAX_BATCH = 4096
ADVANCE = 1
LIVE_TABLES = 2
SCHEDULE_SETTLED = 4

OK = 0
ERR_INVALID_ARG = -1
ERR_FULL = -2
ERR_NOT_ACTIVE = -3
ERR_CAPACITY = -4
ERR_ALIGN = -5
ERR_CUDA = -6
ERR_DEVICE = -7

DEVERR_ROW = 1
DEVERR_COUNT = 2
DEVERR_POSITION = 4
DEVERR_BLOCK = 8
DEVERR_SLOT = 16
DEVERR_TIMEOUT = 32
DEVERR_TABLE_FULL = 64
DEVERR_OUTPUT_FULL = 128
DEVERR_DUP = 256

_NAMES = {OK: "PKV_OK", ERR_INVALID_ARG: "PKV_ERR_INVALID_ARG", ERR_FULL: "PKV_ERR_FULL",
          ERR_NOT_ACTIVE: "PKV_ERR_NOT_ACTIVE", ERR_CAPACITY: "PKV_ERR_CAPACITY",
          ERR_ALIGN: "PKV_ERR_ALIGN", ERR_CUDA: "PKV_ERR_CUDA", ERR_DEVICE: "PKV_ERR_DEVICE"}

# Every symbol the header declares.
EXPORTS = [
    "pkv_state_create", "pkv_state_destroy", "pkv_add_request", "pkv_update_request",
    "pkv_remove_request", "pkv_prepare_batch", "pkv_prepare_batch_device",
    "pkv_prepare_batch_static",
    "pkv_kv_cache_write", "pkv_kv_cache_write_layers", "pkv_kv_cache_write_step",
    "pkv_kv_indices", "pkv_apply_step", "pkv_block_keys", "pkv_prefix_cache_create", "pkv_prefix_cache_destroy",
    "pkv_prefix_cache_insert", "pkv_prefix_cache_match", "pkv_pool_reset", "pkv_pool_size",
    "pkv_pool_read", "pkv_allocate_slots", "pkv_release_blocks", "pkv_get_error",
    "pkv_state_error_word", "pkv_row_info", "pkv_read_row", "pkv_last_cuda_error",
    "pkv_version", "pkv_selftest_wait_timeout",
]


class PkvError(RuntimeError):
    def __init__(self, code: int, call: str):
        extra = ""
        if code == ERR_CUDA and _LIB is not None:
            extra = f" (cudaError {_LIB.pkv_last_cuda_error()})"
        super().__init__(f"{call} failed: {_NAMES.get(code, code)}{extra}")
        self.code = code


class GroupSpec(C.Structure):
    _fields_ = [("block_size", C.c_int32), ("max_blocks_per_req", C.c_int32),
                ("num_blocks", C.c_int64)]


class BatchOut(C.Structure):
    _fields_ = [("index_mapping", C.c_void_p), ("query_start_loc", C.c_void_p),
                ("seq_lens", C.c_void_p), ("positions", C.c_void_p),
                ("input_ids", C.c_void_p), ("block_tables", C.c_void_p * MAX_GROUPS),
                ("slot_mapping", C.c_void_p * MAX_GROUPS)]


class StepDelta(C.Structure):
    _fields_ = [("num_finished", C.c_int32), ("finished_rows", C.c_void_p),
                ("num_new", C.c_int32), ("new_token_offsets", C.c_void_p),
                ("new_token_ids", C.c_void_p), ("new_num_computed", C.c_void_p),
                ("new_block_offsets", C.c_void_p * MAX_GROUPS),
                ("new_block_ids", C.c_void_p * MAX_GROUPS),
                ("num_cached", C.c_int32), ("cached_rows", C.c_void_p),
                ("cached_token_offsets", C.c_void_p), ("cached_token_ids", C.c_void_p),
                ("cached_num_computed", C.c_void_p),
                ("cached_block_offsets", C.c_void_p * MAX_GROUPS),
                ("cached_block_ids", C.c_void_p * MAX_GROUPS)]


class KvItem(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("k_cache", C.c_void_p),
                ("v_cache", C.c_void_p), ("slot_mapping", C.c_void_p), ("num_slots", C.c_int64)]


_P32 = C.POINTER(C.c_int32)
_VP = C.c_void_p
_LIB = None


def _declare(lib):
    i32, i64 = C.c_int32, C.c_int64
    sig = {
        "pkv_state_create": [C.POINTER(_VP), i32, i32, i32, C.POINTER(GroupSpec), i64, _VP],
        "pkv_state_destroy": [_VP],
        "pkv_add_request": [_VP, _P32, i32, i32, C.POINTER(_VP), _P32, _P32, _VP],
        "pkv_update_request": [_VP, i32, C.POINTER(_VP), _P32, _P32, i32, i32, _VP],
        "pkv_remove_request": [_VP, i32, _VP],
        "pkv_prepare_batch": [_VP, _P32, _P32, i32, i32, C.POINTER(BatchOut), _P32, _VP],
        "pkv_prepare_batch_device": [_VP, _VP, _VP, i32, i32, i32, C.POINTER(BatchOut), _VP],
        "pkv_prepare_batch_static": [_VP, _VP, i32, i32, i32, C.POINTER(GroupSpec),
                                     C.POINTER(_VP), _P32, _P32, i32, C.POINTER(BatchOut),
                                     _VP, _P32, _VP],
        "pkv_kv_cache_write": [_VP, _VP, i64, i64, _VP, _VP, i64, i32, _VP, i32, _VP, _VP],
        "pkv_kv_cache_write_layers": [i32, C.POINTER(_VP), C.POINTER(_VP), i64, i64,
                                      C.POINTER(_VP), C.POINTER(_VP), i64, i32, _VP, i32,
                                      _VP, _VP],
        "pkv_kv_cache_write_step": [i32, C.POINTER(KvItem), i64, i64, i32, i32, _VP, _VP],
        "pkv_apply_step": [_VP, C.POINTER(StepDelta), _P32, _VP],
        "pkv_kv_indices": [_VP, i32, _VP, _VP, i32, _VP, _VP, i64, _VP, _VP],
        "pkv_block_keys": [_VP, _P32, i32, i32, _P32, _VP, i64, _VP],
        "pkv_prefix_cache_create": [C.POINTER(_VP), i64, _VP],
        "pkv_prefix_cache_destroy": [_VP],
        "pkv_prefix_cache_insert": [_VP, _VP, _VP, i64, _VP, _VP],
        "pkv_prefix_cache_match": [_VP, _VP, _VP, _VP, i32, _VP, _VP, _VP],
        "pkv_pool_reset": [_VP, i32, _P32, i32, _VP],
        "pkv_pool_size": [_VP, i32, _P32],
        "pkv_pool_read": [_VP, i32, _P32, i32, _VP],
        "pkv_allocate_slots": [_VP, _P32, _P32, _P32, i32, _P32, i32, _P32, _P32, _VP],
        "pkv_release_blocks": [_VP, _P32, i32, _VP],
        "pkv_get_error": [_VP, _P32],
        "pkv_state_error_word": [_VP, C.POINTER(_VP)],
        "pkv_row_info": [_VP, i32, _P32, _P32, _P32, _P32],
        "pkv_read_row": [_VP, i32, _P32, _P32, i32, C.POINTER(_P32), _VP],
        "pkv_last_cuda_error": [],
        "pkv_version": [],
        "pkv_selftest_wait_timeout": [_VP, C.c_uint32, _VP],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = C.c_int
    return lib


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                "paged_kv_prep_gb300: the CUDA library libpkv.so is not built "
                "(run paged_kv_prep_gb300.build.build() or __graft_entry__.build()); "
                "there is no fallback path")
        _LIB = _declare(C.CDLL(LIBRARY))
    return _LIB


def _check(rc, call):
    if rc != OK:
        raise PkvError(rc, call)


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p32(a):
    return a.ctypes.data_as(_P32)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr() if t.numel() else 0)


@dataclass
class Batch:
    """Device outputs of one prepare call (torch tensors)."""

    index_mapping: object
    query_start_loc: object
    seq_lens: object
    positions: object
    input_ids: object
    block_tables: list
    slot_mapping: list
    total_tokens: int

    def struct(self) -> BatchOut:
        o = BatchOut()
        o.index_mapping = self.index_mapping.data_ptr() if self.index_mapping.numel() else None
        o.query_start_loc = self.query_start_loc.data_ptr()
        o.seq_lens = self.seq_lens.data_ptr() if self.seq_lens.numel() else None
        o.positions = self.positions.data_ptr() if self.positions.numel() else None
        o.input_ids = self.input_ids.data_ptr() if self.input_ids.numel() else None
        for g, t in enumerate(self.block_tables):
            o.block_tables[g] = t.data_ptr() if t.numel() else None
        for g, t in enumerate(self.slot_mapping):
            o.slot_mapping[g] = t.data_ptr() if t.numel() else None
        return o


class State:
    """The worker's persistent request-state table on the current CUDA device
    (``pkv_state_create`` ... ``pkv_state_destroy``)."""

    def __init__(self, max_reqs, max_model_len, groups, ring_bytes=0, stream=None):
        """groups: sequence of (block_size, max_blocks_per_req, num_blocks)
        tuples, or objects with those attributes."""
        L = lib()
        specs = []
        for g in groups:
            if isinstance(g, (tuple, list)):
                specs.append(tuple(int(x) for x in g))
            else:
                specs.append((int(g.block_size), int(g.max_blocks_per_req), int(g.num_blocks)))
        self.G = len(specs)
        self.block_size = [s[0] for s in specs]
        self.W = [s[1] for s in specs]
        self.num_blocks = [s[2] for s in specs]
        self.max_reqs = int(max_reqs)
        self.max_model_len = int(max_model_len)
        arr = (GroupSpec * max(self.G, 1))(*[GroupSpec(*s) for s in specs])
        h = C.c_void_p()
        _check(L.pkv_state_create(C.byref(h), self.max_reqs, self.max_model_len, self.G, arr,
                                  int(ring_bytes), _stream(stream)), "pkv_state_create")
        self._h = h

    # -- lifecycle ----------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            _check(lib().pkv_state_destroy(self._h), "pkv_state_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- request state ----------------------------------------------------------
    def _block_args(self, blocks):
        if blocks is None:
            blocks = [()] * self.G
        arrs = [_i32(b) for b in blocks]
        ptrs = (C.c_void_p * max(self.G, 1))(*[a.ctypes.data if a.size else None for a in arrs])
        counts = np.array([a.size for a in arrs], dtype=np.int32)
        return arrs, ptrs, counts

    def add_request(self, token_ids, num_computed, blocks, stream=None, check=True):
        tok = _i32(token_ids)
        arrs, ptrs, counts = self._block_args(blocks)
        row = C.c_int32(-1)
        rc = lib().pkv_add_request(self._h, _p32(tok) if tok.size else None, tok.size,
                                   int(num_computed), ptrs, _p32(counts), C.byref(row),
                                   _stream(stream))
        if check:
            _check(rc, "pkv_add_request")
            return row.value
        return row.value if rc == OK else rc

    def update_request(self, row, new_blocks=None, new_token_ids=(), num_computed=-1,
                       stream=None, check=True):
        tok = _i32(new_token_ids)
        arrs, ptrs, counts = self._block_args(new_blocks)
        rc = lib().pkv_update_request(self._h, int(row), ptrs, _p32(counts),
                                      _p32(tok) if tok.size else None, tok.size,
                                      int(num_computed), _stream(stream))
        if check:
            _check(rc, "pkv_update_request")
        return rc

    def remove_request(self, row, stream=None, check=True):
        rc = lib().pkv_remove_request(self._h, int(row), _stream(stream))
        if check:
            _check(rc, "pkv_remove_request")
        return rc

    def apply_step(self, finished=(), new=(), cached=(), stream=None, check=True):
        """Apply one step's scheduler output (``pkv_apply_step``).

        finished: rows to free; new: (token_ids, num_computed, blocks per
        group) per new request; cached: (row, new_token_ids, num_computed or
        -1, new blocks per group) per cached request.  Returns the new rows."""

        def csr(lists):
            lists = [_i32(x) for x in lists]
            off = np.zeros(len(lists) + 1, np.int32)
            if lists:
                off[1:] = np.cumsum([x.size for x in lists])
            flat = np.concatenate(lists) if lists and off[-1] else np.zeros(0, np.int32)
            return off, flat

        nt_off, nt_ids = csr([x[0] for x in new])
        ct_off, ct_ids = csr([x[1] for x in cached])
        nb = [csr([x[2][g] for x in new]) for g in range(self.G)]
        cb = [csr([x[3][g] for x in cached]) for g in range(self.G)]
        out = self.apply_step_arrays(
            list(finished), nt_off, nt_ids, [x[1] for x in new],
            [b[0] for b in nb], [b[1] for b in nb],
            [x[0] for x in cached], ct_off, ct_ids, [x[2] for x in cached],
            [b[0] for b in cb], [b[1] for b in cb], stream=stream, check=check)
        return out.tolist() if isinstance(out, np.ndarray) else out

    def apply_step_arrays(self, finished_rows, new_token_offsets, new_token_ids,
                          new_num_computed, new_block_offsets, new_block_ids, cached_rows,
                          cached_token_offsets, cached_token_ids, cached_num_computed,
                          cached_block_offsets, cached_block_ids, stream=None, check=True):
        """``pkv_apply_step`` from a scheduler output already packed as int32
        arrays: offsets are CSR ([count + 1], starting at 0) into the flat
        token / block id arrays, block arrays are one per KV-cache group.
        Returns the new requests' rows (int32 numpy array)."""
        keep = []

        def arr(a):
            a = _i32(a)
            keep.append(a)
            return a.ctypes.data if a.size else None

        d = StepDelta()
        fin = _i32(finished_rows)
        d.num_finished = int(fin.size)
        d.finished_rows = arr(fin)
        nnc = _i32(new_num_computed)
        d.num_new = int(nnc.size)
        d.new_token_offsets = arr(new_token_offsets)
        d.new_token_ids = arr(new_token_ids)
        d.new_num_computed = arr(nnc)
        cr = _i32(cached_rows)
        d.num_cached = int(cr.size)
        d.cached_rows = arr(cr)
        d.cached_token_offsets = arr(cached_token_offsets)
        d.cached_token_ids = arr(cached_token_ids)
        d.cached_num_computed = arr(cached_num_computed)
        for g in range(self.G):
            d.new_block_offsets[g] = arr(new_block_offsets[g])
            d.new_block_ids[g] = arr(new_block_ids[g])
            d.cached_block_offsets[g] = arr(cached_block_offsets[g])
            d.cached_block_ids[g] = arr(cached_block_ids[g])
        out = np.zeros(max(d.num_new, 1), np.int32)
        rc = lib().pkv_apply_step(self._h, C.byref(d), _p32(out), _stream(stream))
        if check:
            _check(rc, "pkv_apply_step")
            return out[:d.num_new]
        return rc if rc != OK else out[:d.num_new]

    def block_keys(self, rows, block_size, stream=None):
        """Prefix-cache keys of the full blocks of rows' known tokens
        (``pkv_block_keys``): (host int32 offsets [n+1], device int64 keys,
        the uint64 keys' bits)."""
        import torch

        r = _i32(rows)
        n = int(r.size)
        off = np.zeros(n + 1, np.int32)
        _check(lib().pkv_block_keys(self._h, _p32(r) if n else None, n, int(block_size),
                                    _p32(off), None, 0, _stream(stream)), "pkv_block_keys")
        keys = torch.empty(max(int(off[-1]), 1), dtype=torch.int64, device="cuda")
        _check(lib().pkv_block_keys(self._h, _p32(r) if n else None, n, int(block_size),
                                    _p32(off), C.c_void_p(keys.data_ptr()), int(keys.numel()),
                                    _stream(stream)), "pkv_block_keys")
        return off, keys[: int(off[-1])]

    def block_keys_into(self, rows, block_size, offsets, keys, stream=None):
        """``pkv_block_keys`` into preallocated outputs: rows and offsets
        (int32 numpy, n and n + 1), keys (int64 device tensor)."""
        _check(lib().pkv_block_keys(self._h, _p32(rows), int(rows.size), int(block_size),
                                    _p32(offsets), C.c_void_p(keys.data_ptr()),
                                    int(keys.numel()), _stream_handle(stream)), "pkv_block_keys")

    # -- free-block pools and allocate_slots ---------------------------------
    def pool_reset(self, group, free_ids, stream=None):
        ids = _i32(free_ids)
        _check(lib().pkv_pool_reset(self._h, int(group), _p32(ids) if ids.size else None,
                                    int(ids.size), _stream(stream)), "pkv_pool_reset")

    def pool_size(self, group):
        c = C.c_int32()
        _check(lib().pkv_pool_size(self._h, int(group), C.byref(c)), "pkv_pool_size")
        return c.value

    def pool(self, group, stream=None):
        n = self.pool_size(group)
        out = np.zeros(max(n, 1), np.int32)
        _check(lib().pkv_pool_read(self._h, int(group), _p32(out), n, _stream(stream)),
               "pkv_pool_read")
        return out[:n]

    def allocate_slots(self, rows, num_new, lookahead=None, windows=None, watermark=0,
                       stream=None, check=True):
        """Returns (admitted count, new blocks [n][G])."""
        r = _i32(rows)
        nn = _i32(num_new)
        n = int(r.size)
        la = None if lookahead is None else _i32(lookahead)
        win = None if windows is None else _i32(windows)
        adm = C.c_int32(0)
        nb = np.zeros(max(n * self.G, 1), np.int32)
        rc = lib().pkv_allocate_slots(self._h, _p32(r) if n else None, _p32(nn) if n else None,
                                      _p32(la) if la is not None and n else None, n,
                                      _p32(win) if win is not None else None, int(watermark),
                                      C.byref(adm), _p32(nb), _stream(stream))
        if rc != OK:
            if check:
                raise PkvError(rc, "pkv_allocate_slots")
            return rc
        return adm.value, nb[:n * self.G].reshape(n, self.G)

    def release_blocks(self, rows, stream=None):
        r = _i32(rows)
        _check(lib().pkv_release_blocks(self._h, _p32(r) if r.size else None, int(r.size),
                                        _stream(stream)), "pkv_release_blocks")

    def row_info(self, row):
        a, c, n = C.c_int32(), C.c_int32(), C.c_int32()
        nb = np.zeros(self.G, np.int32)
        _check(lib().pkv_row_info(self._h, int(row), C.byref(a), C.byref(c), C.byref(n),
                                  _p32(nb)), "pkv_row_info")
        return dict(active=bool(a.value), completed=c.value, n_tokens=n.value, num_blocks=nb)

    def read_row(self, row, n_tokens=None, stream=None):
        info = self.row_info(row)
        nt = info["n_tokens"] if n_tokens is None else int(n_tokens)
        tok = np.zeros(max(nt, 1), np.int32)
        tabs = [np.zeros(w, np.int32) for w in self.W]
        tptr = (_P32 * max(self.G, 1))(*[_p32(t) for t in tabs])
        comp = C.c_int32()
        _check(lib().pkv_read_row(self._h, int(row), C.byref(comp), _p32(tok), nt, tptr,
                                  _stream(stream)), "pkv_read_row")
        return dict(completed=comp.value, tokens=tok[:nt], block_table=tabs)

    # -- batch -----------------------------------------------------------------
    def alloc_batch(self, n, total_tokens, device="cuda"):
        import torch

        i32 = dict(dtype=torch.int32, device=device)
        return Batch(
            index_mapping=torch.empty(n, **i32),
            query_start_loc=torch.empty(n + 1, **i32),
            seq_lens=torch.empty(n, **i32),
            positions=torch.empty(total_tokens, **i32),
            input_ids=torch.empty(total_tokens, **i32),
            block_tables=[torch.empty(n, w, **i32) for w in self.W],
            slot_mapping=[torch.empty(total_tokens, dtype=torch.int64, device=device)
                          for _ in self.W],
            total_tokens=int(total_tokens))

    def prepare_batch(self, rows, num_sched, flags=0, out=None, stream=None, check=True):
        """Build the step's batch from host arrays (``pkv_prepare_batch``).
        Returns a Batch of device tensors (allocated unless ``out`` is given)."""
        r = _i32(rows)
        ns = _i32(num_sched)
        n = int(r.size)
        if out is None:
            out = self.alloc_batch(n, int(ns.sum(dtype=np.int64)) if n else 0)
        st = out.struct()
        total = C.c_int32(0)
        rc = lib().pkv_prepare_batch(self._h, _p32(r) if n else None, _p32(ns) if n else None,
                                     n, int(flags), C.byref(st), C.byref(total), _stream(stream))
        if check:
            _check(rc, "pkv_prepare_batch")
        elif rc != OK:
            return rc
        out.total_tokens = total.value
        return out

    def prepare_batch_device(self, d_rows, d_num_sched, total_tokens, out=None, stream=None,
                             check=True, flags=0):
        """Build the step's batch from a schedule already in device memory
        (``pkv_prepare_batch_device``); d_rows / d_num_sched are int32 tensors."""
        n = int(d_rows.numel())
        if out is None:
            out = self.alloc_batch(n, int(total_tokens), device=d_rows.device)
        st = out.struct()
        rc = lib().pkv_prepare_batch_device(self._h, _ptr(d_rows), _ptr(d_num_sched), n,
                                            int(total_tokens), int(flags), C.byref(st),
                                            _stream(stream))
        if check:
            _check(rc, "pkv_prepare_batch_device")
            return out
        return out if rc == OK else rc

    def kv_indices(self, group, index_mapping, seq_lens, capacity=None, out=None,
                   last_page_len=True, stream=None, check=True):
        """Paged (CSR) block table of a prepared batch (``pkv_kv_indices``):
        returns (kv_indptr [n+1], kv_indices [capacity], last_page_len [n] or
        None) as device tensors; the live entries are kv_indices[:kv_indptr[n]].
        ``index_mapping`` / ``seq_lens`` are the batch's int32 device tensors;
        ``out`` may supply the three buffers."""
        import torch

        n = int(index_mapping.numel())
        if capacity is None:
            capacity = n * self.W[group]
        if out is None:
            dev = index_mapping.device
            out = (torch.empty(n + 1, dtype=torch.int32, device=dev),
                   torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev),
                   torch.empty(max(n, 1), dtype=torch.int32, device=dev)
                   if last_page_len else None)
        indptr, indices, last = out
        rc = lib().pkv_kv_indices(self._h, int(group), _ptr(index_mapping), _ptr(seq_lens), n,
                                  _ptr(indptr), _ptr(indices), int(capacity),
                                  _ptr(last) if last is not None else None, _stream(stream))
        if check:
            _check(rc, "pkv_kv_indices")
            return out
        return out if rc == OK else rc

    # -- errors ----------------------------------------------------------------
    def get_error(self) -> int:
        code = C.c_int32(0)
        _check(lib().pkv_get_error(self._h, C.byref(code)), "pkv_get_error")
        return code.value

    @property
    def error_word(self) -> int:
        p = C.c_void_p()
        _check(lib().pkv_state_error_word(self._h, C.byref(p)), "pkv_state_error_word")
        return p.value


def _line_args(k, k_cache):
    line = k_cache[0].numel() * k_cache.element_size() if k_cache.shape[0] else 0
    if k_cache.numel() and not k_cache.is_contiguous():
        raise ValueError("the cache must be contiguous")
    ks = k.stride(0) * k.element_size() if k.dim() >= 1 and k.shape[0] else line
    return line, ks


def kv_cache_write(k, v, k_cache, v_cache, slot_mapping, num_tokens=None, d_error=None,
                   stream=None, check=True):
    """Store each token's K and V line at its slot (``pkv_kv_cache_write``).
    k, v: device tensors whose first dim is the token (row stride allowed, each
    row's line contiguous); k_cache, v_cache: contiguous [num_slots, ...];
    slot_mapping: int64 device tensor."""
    T = int(slot_mapping.numel()) if num_tokens is None else int(num_tokens)
    line, ks = _line_args(k, k_cache)
    _, vs = _line_args(v, v_cache)
    rc = lib().pkv_kv_cache_write(_ptr(k), _ptr(v), ks, vs, _ptr(k_cache), _ptr(v_cache),
                                  int(k_cache.shape[0]), int(line), _ptr(slot_mapping), T,
                                  C.c_void_p(d_error) if d_error else None, _stream(stream))
    if check:
        _check(rc, "pkv_kv_cache_write")
    return rc


def kv_cache_write_layers(ks, vs, k_caches, v_caches, slot_mapping, num_tokens=None,
                          d_error=None, stream=None, check=True):
    """The KV store for several layers sharing one slot_mapping, in one launch
    (``pkv_kv_cache_write_layers``).  Lists of same-shaped tensors."""
    L = len(ks)
    T = int(slot_mapping.numel()) if num_tokens is None else int(num_tokens)
    line, kst = _line_args(ks[0], k_caches[0])
    _, vst = _line_args(vs[0], v_caches[0])
    arr = lambda ts: (C.c_void_p * max(L, 1))(*[t.data_ptr() for t in ts])  # noqa: E731
    rc = lib().pkv_kv_cache_write_layers(L, arr(ks), arr(vs), kst, vst, arr(k_caches),
                                         arr(v_caches), int(k_caches[0].shape[0]), int(line),
                                         _ptr(slot_mapping), T,
                                         C.c_void_p(d_error) if d_error else None,
                                         _stream(stream))
    if check:
        _check(rc, "pkv_kv_cache_write_layers")
    return rc


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


class KvStoreCall:
    """``pkv_kv_cache_write_layers`` with its arguments marshalled once.

    For a step that repeats with the same buffers (the same K/V sources,
    caches and slot_mapping tensors every step), building the pointer arrays
    each call costs more host time than the kernel takes on a small batch;
    this object builds them once and each call only passes the stream."""

    def __init__(self, ks, vs, k_caches, v_caches, slot_mapping, num_tokens=None,
                 d_error=None):
        self._keep = (list(ks), list(vs), list(k_caches), list(v_caches), slot_mapping)
        L = len(ks)
        T = int(slot_mapping.numel()) if num_tokens is None else int(num_tokens)
        line, kst = _line_args(ks[0], k_caches[0])
        _, vst = _line_args(vs[0], v_caches[0])
        arr = lambda ts: (C.c_void_p * max(L, 1))(*[t.data_ptr() for t in ts])  # noqa: E731
        self._args = (L, arr(ks), arr(vs), kst, vst, arr(k_caches), arr(v_caches),
                      int(k_caches[0].shape[0]), int(line), _ptr(slot_mapping), T,
                      C.c_void_p(d_error) if d_error else None)
        self._fn = lib().pkv_kv_cache_write_layers

    def __call__(self, stream=None):
        rc = self._fn(*self._args, _stream_handle(stream))
        if rc != OK:
            raise PkvError(rc, "pkv_kv_cache_write_layers")


class PrepareDeviceCall:
    """``pkv_prepare_batch_device`` with its arguments marshalled once (the
    schedule tensors and the output Batch are reused every call)."""

    def __init__(self, state, d_rows, d_num_sched, total_tokens, out, flags=0):
        self._keep = (state, d_rows, d_num_sched, out)
        self._st = out.struct()
        self._args = (state._h, _ptr(d_rows), _ptr(d_num_sched), int(d_rows.numel()),
                      int(total_tokens), int(flags), C.byref(self._st))
        self._fn = lib().pkv_prepare_batch_device

    def __call__(self, stream=None):
        rc = self._fn(*self._args, _stream_handle(stream))
        if rc != OK:
            raise PkvError(rc, "pkv_prepare_batch_device")


class PrepareHostCall:
    """``pkv_prepare_batch`` (host schedule) with the state and the output
    Batch marshalled once; each call passes only the schedule.  For a worker
    that reuses one set of output buffers every step, this takes the per-call
    Python cost from building the output struct and two pointer objects down
    to two address reads."""

    def __init__(self, state, out, flags=0):
        self._keep = (state, out)
        self._st = out.struct()
        self._total = C.c_int32(0)
        _VPT = C.c_void_p
        proto = C.CFUNCTYPE(C.c_int, _VPT, _VPT, _VPT, C.c_int32, C.c_int32, _VPT, _VPT, _VPT)
        self._fn = proto(("pkv_prepare_batch", lib()))
        self._h = state._h.value if isinstance(state._h, C.c_void_p) else state._h
        self._flags = int(flags)
        self._out_addr = C.addressof(self._st)
        self._total_addr = C.addressof(self._total)
        self._out = out
        # the buffers' capacity: requests and scheduled tokens
        self._cap_n = min(int(out.index_mapping.numel()), int(out.query_start_loc.numel()) - 1)
        self._cap_t = int(out.positions.numel())
        self._last = [None, None]

    def _addr(self, a, which):
        # an int32 contiguous array's address, remembered for the same array
        # object (held here, so it can be neither freed nor resized)
        last = self._last[which]
        if last is not None and last[0] is a:
            return last[1]
        addr = a.ctypes.data
        self._last[which] = (a, addr)
        return addr

    def __call__(self, rows, num_sched, stream=None):
        """Valid while the state is open; the schedule must fit the buffers."""
        r = np.ascontiguousarray(rows, dtype=np.int32)
        ns = np.ascontiguousarray(num_sched, dtype=np.int32)
        n = r.size
        if ns.size != n:
            raise ValueError("rows and num_sched differ in length")
        total = sum(ns.tolist()) if n <= 64 else int(ns.sum(dtype=np.int64))
        if n > self._cap_n or total > self._cap_t:
            raise ValueError("the schedule does not fit the output buffers")
        rp = self._addr(r, 0) if n else None
        np_ = self._addr(ns, 1) if n else None
        rc = self._fn(self._h, rp, np_, n, self._flags, self._out_addr, self._total_addr,
                      _stream_handle(stream))
        if rc != OK:
            raise PkvError(rc, "pkv_prepare_batch")
        self._out.total_tokens = self._total.value
        return self._out


def selftest_wait_timeout(d_error, polls=1000, stream=None):
    """``pkv_selftest_wait_timeout``: a kernel wait that nothing completes
    gives up after ``polls`` polls and ORs PKV_DEVERR_TIMEOUT into d_error
    (an int32 device tensor)."""
    _check(lib().pkv_selftest_wait_timeout(C.c_void_p(d_error.data_ptr()), int(polls),
                                           _stream_handle(stream)), "pkv_selftest_wait_timeout")


def _step_items(items):
    """items: sequence of (k, v, k_cache, v_cache, slot_mapping) tensors."""
    arr = (KvItem * max(len(items), 1))()
    line = kst = vst = None
    for i, (k, v, kc, vc, sm) in enumerate(items):
        ln, ks = _line_args(k, kc)
        _, vs = _line_args(v, vc)
        if line is None:
            line, kst, vst = ln, ks, vs
        elif (ln, ks, vs) != (line, kst, vst):
            raise ValueError("all items of a step share line size and source strides")
        arr[i] = KvItem(k.data_ptr(), v.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                        sm.data_ptr() if sm.numel() else None, int(kc.shape[0]))
    return arr, int(line or 16), int(kst or 16), int(vst or 16)


def kv_cache_write_step(items, num_tokens=None, d_error=None, stream=None, check=True):
    """The step's KV store for several (layer, group) items, each with its own
    slot_mapping and caches, in one launch (``pkv_kv_cache_write_step``)."""
    arr, line, kst, vst = _step_items(items)
    T = int(items[0][4].numel()) if num_tokens is None and items else int(num_tokens or 0)
    rc = lib().pkv_kv_cache_write_step(len(items), arr, kst, vst, line, T,
                                       C.c_void_p(d_error) if d_error else None,
                                       _stream_handle(stream))
    if check and rc != OK:
        raise PkvError(rc, "pkv_kv_cache_write_step")
    return rc


class KvStepCall:
    """``pkv_kv_cache_write_step`` with its arguments marshalled once."""

    def __init__(self, items, num_tokens=None, d_error=None):
        self._keep = [tuple(it) for it in items]
        self._arr, line, kst, vst = _step_items(items)
        T = int(items[0][4].numel()) if num_tokens is None else int(num_tokens)
        self._args = (len(items), self._arr, kst, vst, line, T,
                      C.c_void_p(d_error) if d_error else None)
        self._fn = lib().pkv_kv_cache_write_step

    def __call__(self, stream=None):
        rc = self._fn(*self._args, _stream_handle(stream))
        if rc != OK:
            raise PkvError(rc, "pkv_kv_cache_write_step")


class PrefixCache:
    """Device index of cached blocks, key -> block id (``pkv_prefix_cache_*``)."""

    def __init__(self, capacity, stream=None):
        h = C.c_void_p()
        _check(lib().pkv_prefix_cache_create(C.byref(h), int(capacity), _stream_handle(stream)),
               "pkv_prefix_cache_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _check(lib().pkv_prefix_cache_destroy(self._h), "pkv_prefix_cache_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def insert(self, keys, block_ids, d_error=None, stream=None):
        """keys: int64 device tensor (uint64 bits); block_ids: int32 device tensor."""
        _check(lib().pkv_prefix_cache_insert(self._h, _ptr(keys), _ptr(block_ids),
                                             int(keys.numel()),
                                             C.c_void_p(d_error) if d_error else None,
                                             _stream_handle(stream)), "pkv_prefix_cache_insert")

    def match_into(self, keys, offsets, max_hits, hits, ids, stream=None):
        """``pkv_prefix_cache_match`` into preallocated device tensors."""
        _check(lib().pkv_prefix_cache_match(self._h, _ptr(keys), _ptr(offsets), _ptr(max_hits),
                                            int(max_hits.numel()), _ptr(hits),
                                            C.c_void_p(ids.data_ptr()), _stream_handle(stream)),
               "pkv_prefix_cache_match")

    def match(self, keys, offsets, max_hits, stream=None):
        """Longest cached prefixes: offsets int32 [n+1], max_hits int32 [n]
        (device tensors). Returns (hit_blocks [n], hit_ids like keys)."""
        import torch

        n = int(max_hits.numel())
        hits = torch.empty(n, dtype=torch.int32, device=keys.device)
        ids = torch.empty(max(int(keys.numel()), 1), dtype=torch.int32, device=keys.device)
        _check(lib().pkv_prefix_cache_match(self._h, _ptr(keys), _ptr(offsets), _ptr(max_hits),
                                            n, _ptr(hits), C.c_void_p(ids.data_ptr()),
                                            _stream_handle(stream)), "pkv_prefix_cache_match")
        return hits, ids[: int(keys.numel())]
