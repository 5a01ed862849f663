"""CPU oracle for the paged-KV input-preparation path (ctypes wrapper).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library
(``paged_kv_prep_gb300``) never imports it, and this package never imports the
product library: the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain single-threaded C loops that
restate the definitions on the pages); this module only marshals numpy arrays
in and out.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

OK, BAD_ARG, FULL, NOT_ACTIVE, CAPACITY = 0, 1, 2, 3, 4

_P32 = C.POINTER(C.c_int32)
_P64 = C.POINTER(C.c_int64)
_PU8 = C.POINTER(C.c_uint8)


def _p32(a):
    return a.ctypes.data_as(_P32)


def _declare(lib):
    lib.oracle_state_new.restype = C.c_void_p
    lib.oracle_state_new.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P32, _P32, _P64]
    lib.oracle_state_free.argtypes = [C.c_void_p]
    lib.oracle_state_free.restype = None
    lib.oracle_add_request.argtypes = [C.c_void_p, _P32, C.c_int32, C.c_int32, _P32, _P32, _P32]
    lib.oracle_update_request.argtypes = [C.c_void_p, C.c_int32, _P32, _P32, _P32,
                                          C.c_int32, C.c_int32]
    lib.oracle_remove_request.argtypes = [C.c_void_p, C.c_int32]
    lib.oracle_read_row.argtypes = [C.c_void_p, C.c_int32, _P32, _P32, _P32, _P32, _P32, _P32]
    lib.oracle_prepare_batch.argtypes = [C.c_void_p, _P32, _P32, C.c_int32, C.c_int32,
                                         _P32, _P32, _P32, _P32, _P32,
                                         C.POINTER(_P32), C.POINTER(_P64), _P32]
    lib.oracle_kv_write.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                    C.c_void_p, C.c_void_p, C.c_int64, C.c_int32,
                                    _P64, C.c_int32]
    lib.oracle_kv_indices.argtypes = [C.c_void_p, C.c_int32, _P32, _P32, C.c_int32,
                                      _P32, _P32, C.c_int64, _P32]
    for name in ("oracle_add_request", "oracle_update_request", "oracle_remove_request",
                 "oracle_read_row", "oracle_prepare_batch", "oracle_kv_write",
                 "oracle_kv_indices"):
        getattr(lib, name).restype = C.c_int
    _PU64 = C.POINTER(C.c_uint64)
    lib.oracle_fnv1a64.argtypes = [C.c_void_p, C.c_int64]
    lib.oracle_fnv1a64.restype = C.c_uint64
    lib.oracle_block_keys.argtypes = [_P32, C.c_int32, C.c_int32, _PU64]
    lib.oracle_block_keys.restype = C.c_int
    lib.oracle_row_block_keys.argtypes = [C.c_void_p, C.c_int32, C.c_int32, _PU64, _P32]
    lib.oracle_row_block_keys.restype = C.c_int
    lib.oracle_prefix_hits.argtypes = [_PU64, C.c_int32, C.c_int32, _PU64, _P32, C.c_int64, _P32]
    lib.oracle_prefix_hits.restype = C.c_int32
    lib.oracle_pool_reset.argtypes = [C.c_void_p, C.c_int32, _P32, C.c_int32]
    lib.oracle_pool_reset.restype = C.c_int
    lib.oracle_pool_count.argtypes = [C.c_void_p, C.c_int32]
    lib.oracle_pool_count.restype = C.c_int32
    lib.oracle_pool_read.argtypes = [C.c_void_p, C.c_int32, _P32]
    lib.oracle_pool_read.restype = None
    lib.oracle_allocate_slots.argtypes = [C.c_void_p, _P32, _P32, _P32, C.c_int32, _P32,
                                          C.c_int32, _P32, _P32]
    lib.oracle_allocate_slots.restype = C.c_int
    lib.oracle_release_blocks.argtypes = [C.c_void_p, _P32, C.c_int32]
    lib.oracle_release_blocks.restype = C.c_int
    return lib


_DEFAULT = None


def load(path: str | None = None):
    """Load the oracle library (building the default one if needed)."""
    global _DEFAULT
    if path is None:
        if _DEFAULT is None:
            _DEFAULT = _declare(C.CDLL(_build.build()))
        return _DEFAULT
    return _declare(C.CDLL(os.path.abspath(path)))


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"oracle {what}: status {code}")
        self.code = code


class OracleState:
    """The worker's request-state table, as the oracle keeps it."""

    def __init__(self, max_reqs, max_model_len, groups, lib=None):
        """groups: sequence of (block_size, max_blocks_per_req, num_blocks)."""
        self.lib = lib if lib is not None else load()
        self.G = len(groups)
        self.block_size = [int(g[0]) for g in groups]
        self.W = [int(g[1]) for g in groups]
        self.max_reqs = int(max_reqs)
        self.max_model_len = int(max_model_len)
        bs = np.array(self.block_size, np.int32)
        W = np.array(self.W, np.int32)
        nb = np.array([int(g[2]) for g in groups], np.int64)
        self._h = self.lib.oracle_state_new(max_reqs, max_model_len, self.G, _p32(bs),
                                            _p32(W), nb.ctypes.data_as(_P64))
        if not self._h:
            raise OracleError(BAD_ARG, "state_new")

    def close(self):
        if self._h:
            self.lib.oracle_state_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _blocks(self, blocks):
        blocks = [np.ascontiguousarray(b, dtype=np.int32) for b in blocks]
        counts = np.array([len(b) for b in blocks], np.int32)
        flat = np.concatenate(blocks) if sum(counts) else np.zeros(1, np.int32)
        return np.ascontiguousarray(flat, np.int32), counts

    def add_request(self, token_ids, num_computed, blocks, check=True):
        tok = np.ascontiguousarray(token_ids, dtype=np.int32)
        if tok.size == 0:
            tok = np.zeros(1, np.int32)
            ntok = 0
        else:
            ntok = tok.size
        flat, counts = self._blocks(blocks)
        row = C.c_int32(-1)
        rc = self.lib.oracle_add_request(self._h, _p32(tok), ntok, int(num_computed),
                                         _p32(flat), _p32(counts), C.byref(row))
        if check and rc != OK:
            raise OracleError(rc, "add_request")
        return row.value if rc == OK else -rc

    def update_request(self, row, new_blocks=None, new_token_ids=(), num_computed=-1,
                       check=True):
        if new_blocks is None:
            new_blocks = [np.zeros(0, np.int32)] * self.G
        flat, counts = self._blocks(new_blocks)
        tok = np.ascontiguousarray(new_token_ids, dtype=np.int32)
        ntok = tok.size
        if ntok == 0:
            tok = np.zeros(1, np.int32)
        rc = self.lib.oracle_update_request(self._h, int(row), _p32(flat), _p32(counts),
                                            _p32(tok), ntok, int(num_computed))
        if check and rc != OK:
            raise OracleError(rc, "update_request")
        return rc

    def remove_request(self, row, check=True):
        rc = self.lib.oracle_remove_request(self._h, int(row))
        if check and rc != OK:
            raise OracleError(rc, "remove_request")
        return rc

    # -- block pools and allocate_slots ------------------------------------
    def pool_reset(self, group, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        rc = self.lib.oracle_pool_reset(self._h, int(group), _p32(ids if ids.size else
                                                                  np.zeros(1, np.int32)),
                                        int(ids.size))
        if rc != OK:
            raise OracleError(rc, "pool_reset")

    def pool(self, group):
        n = self.lib.oracle_pool_count(self._h, int(group))
        out = np.zeros(max(n, 1), np.int32)
        self.lib.oracle_pool_read(self._h, int(group), _p32(out))
        return out[:n]

    def allocate_slots(self, rows, num_new, lookahead=None, windows=None, watermark=0,
                       check=True):
        """Returns (admitted count, new blocks per request per group)."""
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        nn = np.ascontiguousarray(num_new, dtype=np.int32)
        n = int(rows.size)
        la = None if lookahead is None else np.ascontiguousarray(lookahead, dtype=np.int32)
        win = None if windows is None else np.ascontiguousarray(windows, dtype=np.int32)
        adm = C.c_int32(0)
        nb = np.zeros(max(n * self.G, 1), np.int32)
        z = np.zeros(1, np.int32)
        rc = self.lib.oracle_allocate_slots(self._h, _p32(rows if n else z), _p32(nn if n else z),
                                            _p32(la) if la is not None and n else None, n,
                                            _p32(win) if win is not None else None,
                                            int(watermark), C.byref(adm), _p32(nb))
        if rc != OK:
            if check:
                raise OracleError(rc, "allocate_slots")
            return rc
        return adm.value, nb[:n * self.G].reshape(n, self.G)

    def release_blocks(self, rows):
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        rc = self.lib.oracle_release_blocks(self._h, _p32(rows if rows.size else
                                                          np.zeros(1, np.int32)), int(rows.size))
        if rc != OK:
            raise OracleError(rc, "release_blocks")

    def read_row(self, row):
        a, c, n = C.c_int32(), C.c_int32(), C.c_int32()
        nblk = np.zeros(self.G, np.int32)
        bt = np.zeros(sum(self.W), np.int32)
        rc = self.lib.oracle_read_row(self._h, int(row), C.byref(a), C.byref(c), C.byref(n),
                                      None, _p32(nblk), _p32(bt))
        if rc != OK:
            raise OracleError(rc, "read_row")
        tok = np.zeros(max(n.value, 1), np.int32)
        self.lib.oracle_read_row(self._h, int(row), C.byref(a), C.byref(c), C.byref(n),
                                 _p32(tok), None, None)
        lines, off = [], 0
        for w in self.W:
            lines.append(bt[off:off + w].copy())
            off += w
        return dict(active=bool(a.value), completed=c.value, tokens=tok[:n.value].copy(),
                    num_blocks=nblk, block_table=lines)

    def prepare_batch(self, rows, num_sched, advance=False, check=True):
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        ns = np.ascontiguousarray(num_sched, dtype=np.int32)
        n = int(rows.size)
        T = int(ns.sum()) if n else 0
        im = np.zeros(max(n, 1), np.int32)
        qsl = np.zeros(n + 1, np.int32)
        sl = np.zeros(max(n, 1), np.int32)
        pos = np.zeros(max(T, 1), np.int32)
        ids = np.zeros(max(T, 1), np.int32)
        bts = [np.zeros(max(n, 1) * w, np.int32) for w in self.W]
        slots = [np.zeros(max(T, 1), np.int64) for _ in self.W]
        bt_ptrs = (_P32 * self.G)(*[_p32(b) for b in bts])
        sl_ptrs = (_P64 * self.G)(*[s.ctypes.data_as(_P64) for s in slots])
        total = C.c_int32(0)
        rows_a = rows if n else np.zeros(1, np.int32)
        ns_a = ns if n else np.zeros(1, np.int32)
        rc = self.lib.oracle_prepare_batch(self._h, _p32(rows_a), _p32(ns_a), n,
                                           1 if advance else 0, _p32(im), _p32(qsl),
                                           _p32(sl), _p32(pos), _p32(ids), bt_ptrs, sl_ptrs,
                                           C.byref(total))
        if rc != OK:
            if check:
                raise OracleError(rc, "prepare_batch")
            return rc
        T = total.value
        return dict(
            index_mapping=im[:n], query_start_loc=qsl, seq_lens=sl[:n],
            positions=pos[:T], input_ids=ids[:T],
            block_tables=[b[:n * w].reshape(n, w) for b, w in zip(bts, self.W)],
            slot_mapping=[s[:T] for s in slots], total_tokens=T)

    def kv_indices(self, group, index_mapping, seq_lens, capacity=None, check=True):
        """Paged (CSR) block table of a prepared batch for one group:
        (kv_indptr [n+1], kv_indices [kv_indptr[n]], last_page_len [n])."""
        im = np.ascontiguousarray(index_mapping, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        n = int(im.size)
        if capacity is None:
            capacity = n * self.W[group]
        indptr = np.zeros(n + 1, np.int32)
        indices = np.zeros(max(int(capacity), 1), np.int32)
        last = np.zeros(max(n, 1), np.int32)
        z = np.zeros(1, np.int32)
        rc = self.lib.oracle_kv_indices(self._h, int(group), _p32(im if n else z),
                                        _p32(sl if n else z), n, _p32(indptr), _p32(indices),
                                        int(capacity), _p32(last))
        if rc != OK:
            if check:
                raise OracleError(rc, "kv_indices")
            return rc
        return indptr, indices[:indptr[n]].copy(), last[:n].copy()


def kv_write(k, v, k_cache, v_cache, slot_mapping, lib=None):
    """Store each token's K and V line at its slot.  k, v: uint8 arrays
    [T, >=line] (row stride taken from the array); caches: uint8 [num_slots,
    line], modified in place.  Returns the status code."""
    lib = lib if lib is not None else load()
    k = np.asarray(k)
    v = np.asarray(v)
    slot = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = int(slot.size)
    line = int(k_cache.shape[1])
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    ks = int(k.strides[0]) if k.ndim == 2 and T else line
    vs = int(v.strides[0]) if v.ndim == 2 and T else line
    assert k.ndim == 2 and k.strides[1] == 1 and v.strides[1] == 1
    return lib.oracle_kv_write(k.ctypes.data, v.ctypes.data, ks, vs, k_cache.ctypes.data,
                               v_cache.ctypes.data, int(k_cache.shape[0]), line,
                               slot.ctypes.data_as(_P64) if T else None, T)


# ---------------------------------------------------------------------------
# prefix-cache block keys
# ---------------------------------------------------------------------------
_PU64 = C.POINTER(C.c_uint64)


def fnv1a64(data: bytes, lib=None) -> int:
    lib = lib if lib is not None else load()
    buf = (C.c_uint8 * max(len(data), 1)).from_buffer_copy(data or b"\0")
    return int(lib.oracle_fnv1a64(buf, len(data)))


def block_keys(token_ids, block_size, lib=None) -> np.ndarray:
    """uint64 keys of the full blocks of token_ids (block + prefix chained)."""
    lib = lib if lib is not None else load()
    tok = np.ascontiguousarray(token_ids, dtype=np.int32)
    n = int(tok.size)
    nfull = n // block_size if block_size > 0 else 0
    # one guard slot past the full blocks: a partial block must get no key
    guard = np.uint64(0x5A5A5A5A5A5A5A5A)
    keys = np.full(nfull + 1, guard, np.uint64)
    rc = lib.oracle_block_keys(_p32(tok if n else np.zeros(1, np.int32)), n, int(block_size),
                               keys.ctypes.data_as(_PU64))
    if rc != OK:
        raise OracleError(rc, "block_keys")
    if keys[nfull] != guard:
        raise OracleError(BAD_ARG, "block_keys wrote a key past the full blocks")
    return keys[:nfull]


def prefix_hits(keys, n_tokens, block_size, index, lib=None):
    """(hit_blocks, hit_ids) for one request against {key: block_id}."""
    lib = lib if lib is not None else load()
    keys = np.ascontiguousarray(keys, dtype=np.uint64)
    ik = np.array(list(index.keys()) or [0], dtype=np.uint64)
    iv = np.array(list(index.values()) or [0], dtype=np.int32)
    out = np.full(max(keys.size, 1), -1, np.int32)
    k = lib.oracle_prefix_hits(keys.ctypes.data_as(_PU64) if keys.size else None, int(n_tokens),
                               int(block_size), ik.ctypes.data_as(_PU64), _p32(iv),
                               len(index), _p32(out))
    return int(k), out[:k].copy()
