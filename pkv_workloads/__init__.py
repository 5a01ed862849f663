"""Seeded synthetic workloads for the paged-KV input-preparation path.

Test and benchmark infrastructure, not part of the library: the tests, the
benchmark and ``smoke()`` share it.  It only decides *what the inputs are*:
which requests exist, in which order they are added to and removed from the
request-state pool, their token ids, the physical
block ids a scheduler would have handed them, the step's schedule (request,
num_scheduled_tokens) and the K/V source bytes.  It contains none of the path's
own arithmetic (no sorting into a batch, no prefix sums, no position or slot
computation, no gathering): those live in the CUDA library and, independently,
in the CPU oracle.

Five workload families follow the five synthetic configurations this library is
measured on (tiny, decode-heavy, mixed chunked prefill, two KV-cache groups,
large 80-layer step).  Every builder takes a seed and size knobs whose defaults
are the full-size configuration; the tests pass smaller values to get cases the
oracle finishes in seconds.

Readings used to turn the configuration text into concrete inputs:

* "context length" is the request's sequence length *after* this step.  A
  decode request with context L has ``L - 1`` computed tokens and schedules 1;
  a prefill chunk of c tokens on a request of context L has ``L - c`` computed
  tokens (the tiny workload's prefills start at position 0).
* A request holds every token id up to ``computed + scheduled`` (prompt plus
  sampled tokens), and physical blocks covering those positions.
* The null block id is -1.  A sliding-window group marks the logical blocks
  that lie wholly before ``max(0, computed - (window - 1))`` as -1, as a
  scheduler that frees out-of-window blocks would ("allocate_slots()" section
  of "从源码读 vLLM Scheduler").
* In the large step, the physical pool of each layer is far smaller than the
  sum of all contexts.  The blocks that receive this step's writes are
  distinct (a random permutation of the pool); older full blocks are drawn
  uniformly from the rest of the pool and may be shared between requests, the
  way prefix-cache hits share blocks.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

TOKEN_VOCAB = 128000

KV_DTYPE_BYTES = {"float16": 2, "bfloat16": 2, "float8_e4m3fn": 1}


@dataclass
class GroupSpec:
    """One KV-cache group: its block size, block-table width and pool size."""

    block_size: int
    max_blocks_per_req: int
    num_blocks: int
    sliding_window: int = 0  # 0 = full attention


@dataclass
class Request:
    """A request as the scheduler hands it to the worker on first sight."""

    handle: int
    token_ids: np.ndarray  # int32, every known token id (prompt + sampled)
    num_computed: int
    blocks: list  # per group: int32 array of physical block ids (-1 = freed)


@dataclass
class Workload:
    name: str
    seed: int
    max_reqs: int
    max_model_len: int
    groups: list
    num_heads: int
    head_dim: int
    kv_dtype: str
    num_layers: int
    # ("add", Request) or ("remove", handle), applied in order to an empty pool
    ops: list = field(default_factory=list)
    # (handle, num_scheduled_tokens) in schedule-output order
    schedule: list = field(default_factory=list)

    @property
    def elem_size(self) -> int:
        return KV_DTYPE_BYTES[self.kv_dtype]

    @property
    def line_bytes(self) -> int:
        """Bytes of one token's K (or V) vectors over all KV heads."""
        return self.num_heads * self.head_dim * self.elem_size

    @property
    def num_sched(self) -> np.ndarray:
        return np.array([c for _, c in self.schedule], dtype=np.int32)

    @property
    def total_tokens(self) -> int:
        return int(sum(c for _, c in self.schedule))

    @property
    def num_scheduled_requests(self) -> int:
        return len(self.schedule)

    def requests(self) -> dict:
        """handle -> Request for every request added by ``ops``."""
        return {r.handle: r for kind, r in self.ops if kind == "add"}


def _blocks_to_cover(num_positions: int, block_size: int) -> int:
    # how many blocks a scheduler allocates for positions [0, num_positions)
    return -(-num_positions // block_size)


def _tokens(rng, length):
    return rng.integers(0, TOKEN_VOCAB, size=length, dtype=np.int32)


def _churn_then_add(rng, handles_to_add, rows, start_handle):
    """Fill every row with an empty dummy request, remove a random subset of
    them as large as the real batch, then add the real requests, so that they
    land on scattered recycled rows."""
    ops = []
    dummies = []
    for k in range(rows):
        h = start_handle + k
        dummies.append(h)
        ops.append(("add", None, h))
    victims = rng.choice(len(dummies), size=len(handles_to_add), replace=False)
    for v in victims:
        ops.append(("remove", None, dummies[int(v)]))
    return ops


def _dummy(handle, num_groups):
    return Request(handle, np.zeros(0, np.int32), 0,
                   [np.zeros(0, np.int32) for _ in range(num_groups)])


def _finish_ops(churn, dummies_groups, reqs, rng, shuffle_adds=False):
    ops = []
    for kind, _, h in churn:
        if kind == "add":
            ops.append(("add", _dummy(h, dummies_groups)))
        else:
            ops.append(("remove", h))
    order = list(range(len(reqs)))
    if shuffle_adds:
        rng.shuffle(order)
    for i in order:
        ops.append(("add", reqs[i]))
    return ops


def _schedule(rng, reqs, nsched):
    order = rng.permutation(len(reqs))
    return [(reqs[int(i)].handle, int(nsched[int(i)])) for i in order]


# --------------------------------------------------------------------------
# tiny: 32-row table, 8 requests, bs 16, 256 blocks, fp16 H8 x D128
# --------------------------------------------------------------------------
def tiny(seed: int = 0) -> Workload:
    rng = np.random.default_rng([seed, 0])
    bs, W, pool, rows, max_len = 16, 16, 256, 32, 256
    while True:
        dec_ctx = rng.integers(1, 201, size=4)
        pre_n = rng.integers(2, 65, size=4)
        if 4 + int(pre_n.sum()) <= 256:
            break
    perm = rng.permutation(pool).astype(np.int32)
    nxt = 0
    reqs, nsched = [], []
    for k in range(8):
        if k < 4:
            L, n = int(dec_ctx[k]), 1
        else:
            n = int(pre_n[k - 4])
            L = n  # prefill from position 0
        nb = _blocks_to_cover(L, bs)
        blocks = perm[nxt:nxt + nb].copy()
        nxt += nb
        reqs.append(Request(1000 + k, _tokens(rng, L), L - n, [blocks]))
        nsched.append(n)
    churn = _churn_then_add(rng, reqs, rows, start_handle=0)
    wl = Workload("tiny", seed, rows, max_len, [GroupSpec(bs, W, pool)], 8, 128,
                  "float16", 1)
    wl.ops = _finish_ops(churn, 1, reqs, rng, shuffle_adds=True)
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


# --------------------------------------------------------------------------
# decode-heavy: 256 decode requests, contexts U[1, 8192], bs 16, W 512
# --------------------------------------------------------------------------
def decode_heavy(seed: int = 0, num_requests: int = 256, max_ctx: int = 8192,
                 pool: int = 131072) -> Workload:
    rng = np.random.default_rng([seed, 1])
    bs = 16
    W = _blocks_to_cover(max_ctx, bs)
    perm = rng.permutation(pool).astype(np.int32)
    nxt = 0
    reqs, nsched = [], []
    ctx = rng.integers(1, max_ctx + 1, size=num_requests)
    for k in range(num_requests):
        L = int(ctx[k])
        nb = _blocks_to_cover(L, bs)
        reqs.append(Request(k, _tokens(rng, L), L - 1, [perm[nxt:nxt + nb].copy()]))
        nxt += nb
        nsched.append(1)
    wl = Workload("decode_heavy", seed, num_requests, max_ctx,
                  [GroupSpec(bs, W, pool)], 8, 128, "bfloat16", 1)
    order = rng.permutation(num_requests)
    wl.ops = [("add", reqs[int(i)]) for i in order]
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


# --------------------------------------------------------------------------
# mixed chunked prefill: budget 8192 = 64 decodes + prefill chunks U[512,2048]
# --------------------------------------------------------------------------
def mixed_prefill(seed: int = 0, budget: int = 8192, num_decode: int = 64,
                  chunk_lo: int = 512, chunk_hi: int = 2048, max_ctx: int = 16384,
                  rows: int = 1024, pool: int = 131072) -> Workload:
    rng = np.random.default_rng([seed, 2])
    bs = 16
    W = _blocks_to_cover(max_ctx, bs)
    chunks = []
    left = budget - num_decode
    while left > 0:
        c = min(int(rng.integers(chunk_lo, chunk_hi + 1)), left)
        chunks.append(c)
        left -= c
    perm = rng.permutation(pool).astype(np.int32)
    nxt = 0
    reqs, nsched = [], []
    h = rows  # handles above the dummies
    for k in range(num_decode):
        L = int(rng.integers(1, max_ctx + 1))
        nb = _blocks_to_cover(L, bs)
        reqs.append(Request(h, _tokens(rng, L), L - 1, [perm[nxt:nxt + nb].copy()]))
        nxt += nb
        h += 1
        nsched.append(1)
    for c in chunks:
        L = int(rng.integers(c, max_ctx + 1))
        nb = _blocks_to_cover(L, bs)
        reqs.append(Request(h, _tokens(rng, L), L - c, [perm[nxt:nxt + nb].copy()]))
        nxt += nb
        h += 1
        nsched.append(c)
    if len(reqs) > rows:
        raise ValueError("more requests than rows")
    churn = _churn_then_add(rng, reqs, rows, start_handle=0)
    wl = Workload("mixed_prefill", seed, rows, max_ctx, [GroupSpec(bs, W, pool)],
                  8, 128, "bfloat16", 1)
    wl.ops = _finish_ops(churn, 1, reqs, rng, shuffle_adds=True)
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


# --------------------------------------------------------------------------
# two KV-cache groups: full attention + sliding window 4096, 1024 requests
# --------------------------------------------------------------------------
def two_groups(seed: int = 0, num_requests: int = 1024, prefill_frac: float = 0.1,
               chunk_hi: int = 256, max_ctx: int = 32768, window: int = 4096) -> Workload:
    rng = np.random.default_rng([seed, 3])
    bs = 16
    W = _blocks_to_cover(max_ctx, bs)
    num_prefill = int(round(prefill_frac * num_requests))
    kinds = np.array([1] * num_prefill + [0] * (num_requests - num_prefill))
    rng.shuffle(kinds)
    specs = []  # (L, n)
    for k in range(num_requests):
        ctx = int(rng.integers(1, max_ctx + 1))
        if kinds[k]:
            n = int(rng.integers(1, chunk_hi + 1))
            L = max(ctx, n)
        else:
            n, L = 1, ctx
        specs.append((L, n))
    # group 0 keeps every block; group 1 frees blocks wholly before the window
    need0, need1 = [], []
    for L, n in specs:
        nb = _blocks_to_cover(L, bs)
        first_kept = max(0, (L - n) - (window - 1)) // bs
        need0.append(nb)
        need1.append((first_kept, nb))
    pool0 = int(sum(need0))
    pool1 = int(sum(nb - f for f, nb in need1))
    perm0 = rng.permutation(pool0).astype(np.int32)
    perm1 = rng.permutation(pool1).astype(np.int32)
    n0 = n1 = 0
    reqs, nsched = [], []
    for k, (L, n) in enumerate(specs):
        b0 = perm0[n0:n0 + need0[k]].copy()
        n0 += need0[k]
        first_kept, nb = need1[k]
        b1 = np.full(nb, -1, np.int32)
        b1[first_kept:] = perm1[n1:n1 + nb - first_kept]
        n1 += nb - first_kept
        reqs.append(Request(k, _tokens(rng, L), L - n, [b0, b1]))
        nsched.append(n)
    groups = [GroupSpec(bs, W, pool0), GroupSpec(bs, W, pool1, sliding_window=window)]
    wl = Workload("two_groups", seed, num_requests, max_ctx, groups, 8, 128,
                  "bfloat16", 1)
    order = rng.permutation(num_requests)
    wl.ops = [("add", reqs[int(i)]) for i in order]
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


# --------------------------------------------------------------------------
# large step: budget 16384 over 4096 requests, bs 32, W 4096, fp8, 80 layers
# --------------------------------------------------------------------------
def large_step(seed: int = 0, num_requests: int = 4096, budget: int = 16384,
               chunk_hi: int = 4096, max_ctx: int = 131072, num_layers: int = 80,
               pool: int = 28610) -> Workload:
    rng = np.random.default_rng([seed, 4])
    bs = 32
    W = _blocks_to_cover(max_ctx, bs)
    log2_max = float(np.log2(max_ctx))
    # prefill chunks until the decodes plus the chunks fill the budget
    chunks = []
    while (num_requests - len(chunks)) + sum(chunks) < budget:
        chunks.append(int(rng.integers(1, chunk_hi + 1)))
    overshoot = (num_requests - len(chunks)) + sum(chunks) - budget
    chunks[-1] -= overshoot
    if chunks and chunks[-1] < 1:
        raise ValueError("budget cannot be met with these sizes")
    num_prefill = len(chunks)
    kinds = np.array([1] * num_prefill + [0] * (num_requests - num_prefill))
    rng.shuffle(kinds)
    ci = 0
    specs = []
    for k in range(num_requests):
        L = int(np.floor(2.0 ** rng.uniform(0.0, log2_max)))
        L = min(max(L, 1), max_ctx)
        if kinds[k]:
            n = chunks[ci]
            ci += 1
            L = max(L, n)
        else:
            n = 1
        specs.append((L, n))
    # blocks written this step: distinct, from a permutation of the pool;
    # older full blocks: uniform over the rest of the pool (may repeat)
    perm = rng.permutation(pool).astype(np.int32)
    nxt = 0
    write_sets = []
    for L, n in specs:
        first_w = (L - n) // bs
        nb = _blocks_to_cover(L, bs)
        write_sets.append((first_w, nb))
        nxt += nb - first_w
    if nxt > pool:
        raise ValueError("pool too small for this step's writes")
    rest = perm[nxt:]
    nxt = 0
    reqs, nsched = [], []
    for k, (L, n) in enumerate(specs):
        first_w, nb = write_sets[k]
        blocks = np.empty(nb, np.int32)
        if first_w:
            if len(rest) == 0:
                raise ValueError("no pool left for history blocks")
            blocks[:first_w] = rest[rng.integers(0, len(rest), size=first_w)]
        blocks[first_w:] = perm[nxt:nxt + nb - first_w]
        nxt += nb - first_w
        reqs.append(Request(k, _tokens(rng, L), L - n, [blocks]))
        nsched.append(n)
    wl = Workload("large_step", seed, num_requests, max_ctx, [GroupSpec(bs, W, pool)],
                  8, 128, "float8_e4m3fn", num_layers)
    order = rng.permutation(num_requests)
    wl.ops = [("add", reqs[int(i)]) for i in order]
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


def decode_large(seed: int = 0, num_requests: int = 4096, max_ctx: int = 2048,
                 width: int = 4096) -> Workload:
    """A pure decode step with the large step's request count and table
    width: 4096 decodes, context U[1, 2048], bs 16, W 4096 (134 MB of table
    rows read and written, as R4's full-row gather asks); the pool is just
    large enough for every request's own blocks, and the K/V lines are one
    bf16 head of 128 (256 bytes), so the one-layer caches take about 2.2 GB.
    Not one of the five configurations: it sizes the decode-only batch build
    at scale."""
    rng = np.random.default_rng([seed, 6])
    bs = 16
    ctx = rng.integers(1, max_ctx + 1, size=num_requests)
    nbs = [_blocks_to_cover(int(L), bs) for L in ctx]
    pool = sum(nbs) + 1024
    perm = rng.permutation(pool).astype(np.int32)
    nxt = 0
    reqs, nsched = [], []
    for k in range(num_requests):
        L, nb = int(ctx[k]), nbs[k]
        reqs.append(Request(k, _tokens(rng, L), L - 1, [perm[nxt:nxt + nb].copy()]))
        nxt += nb
        nsched.append(1)
    wl = Workload("decode_large", seed, num_requests, max_ctx,
                  [GroupSpec(bs, width, pool)], 1, 128, "bfloat16", 1)
    order = rng.permutation(num_requests)
    wl.ops = [("add", reqs[int(i)]) for i in order]
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


BUILDERS = {
    "tiny": tiny,
    "decode_heavy": decode_heavy,
    "decode_large": decode_large,
    "mixed_prefill": mixed_prefill,
    "two_groups": two_groups,
    "large_step": large_step,
}


def build(name: str, seed: int = 0, **kw) -> Workload:
    return BUILDERS[name](seed=seed, **kw)


# --------------------------------------------------------------------------
# K/V source bytes
# --------------------------------------------------------------------------
def kv_sources(wl: Workload, layer: int, group: int, device="cpu", row_pad: int = 0,
               num_tokens: int | None = None):
    """K and V vectors of this step's tokens for one (layer, group): N(0,1)
    drawn in fp32 and cast to the KV dtype, returned as uint8 views of shape
    [T, line_bytes] (row stride ``line_bytes + row_pad`` bytes when row_pad is
    non-zero, as when K and V are slices of a wider fused projection)."""
    import torch

    T = wl.total_tokens if num_tokens is None else num_tokens
    line = wl.line_bytes
    dt = getattr(torch, wl.kv_dtype)
    g = torch.Generator(device=device)
    g.manual_seed(int(wl.seed) * 1_000_003 + layer * 97 + group)
    out = []
    for _ in range(2):
        vals = torch.randn(T, wl.num_heads * wl.head_dim, generator=g, device=device,
                           dtype=torch.float32).to(dt)
        raw = vals.view(torch.uint8)
        if row_pad:
            wide = torch.zeros(T, line + row_pad, dtype=torch.uint8, device=device)
            wide[:, :line] = raw
            raw = wide[:, :line]
        out.append(raw)
    return out[0], out[1]


def all_byte_values_source(num_tokens: int, line_bytes: int, device="cpu", shift: int = 0):
    """A source whose bytes run through all 256 values (every fp8 bit pattern,
    NaNs included), so a byte-exact copy can be told from a float round trip."""
    import torch

    idx = torch.arange(num_tokens * line_bytes, device=device, dtype=torch.int64)
    return ((idx + shift) % 256).to(torch.uint8).view(num_tokens, line_bytes)


# --------------------------------------------------------------------------
# small random states for pins and edge cases
# --------------------------------------------------------------------------
def random_small(seed: int = 0, num_requests: int = 12, block_sizes=(16,),
                 max_ctx: int = 200, max_chunk: int = 40, decode_frac: float = 0.5,
                 rows: int | None = None, churn: bool = True,
                 window: int = 0) -> Workload:
    """A small random step over any block sizes (including 1 and sizes that are
    not powers of two), optionally with a sliding-window last group and with
    requests added onto recycled rows."""
    rng = np.random.default_rng([seed, 5])
    G = len(block_sizes)
    rows = rows if rows is not None else 2 * num_requests
    specs = []
    for _ in range(num_requests):
        if rng.uniform() < decode_frac:
            L = int(rng.integers(1, max_ctx + 1))
            n = 1
        else:
            n = int(rng.integers(1, max_chunk + 1))
            L = int(rng.integers(n, max(n, max_ctx) + 1))
        specs.append((L, n))
    groups, perms, used = [], [], []
    for g, bs in enumerate(block_sizes):
        W = _blocks_to_cover(max(max_ctx, max_chunk), bs) + int(rng.integers(0, 3))
        pool = sum(_blocks_to_cover(L, bs) for L, _ in specs) + int(rng.integers(0, 50))
        sw = window if (window and g == G - 1) else 0
        groups.append(GroupSpec(bs, W, pool, sliding_window=sw))
        perms.append(rng.permutation(pool).astype(np.int32))
        used.append(0)
    reqs, nsched = [], []
    for k, (L, n) in enumerate(specs):
        blocks = []
        for g, spec in enumerate(groups):
            nb = _blocks_to_cover(L, spec.block_size)
            b = perms[g][used[g]:used[g] + nb].copy()
            used[g] += nb
            if spec.sliding_window:
                first_kept = max(0, (L - n) - (spec.sliding_window - 1)) // spec.block_size
                b[:first_kept] = -1
            blocks.append(b)
        reqs.append(Request(rows + k, _tokens(rng, L), L - n, blocks))
        nsched.append(n)
    max_len = max(max_ctx, max_chunk)
    wl = Workload("random_small", seed, rows, max_len, groups, 2, 16, "float16", 1)
    if churn:
        ch = _churn_then_add(rng, reqs, rows, start_handle=0)
        wl.ops = _finish_ops(ch, G, reqs, rng, shuffle_adds=True)
    else:
        wl.ops = [("add", r) for r in reqs]
    wl.schedule = _schedule(rng, reqs, nsched)
    return wl


def apply_ops(state, wl: Workload) -> dict:
    """Replay the workload's add/remove program on a state object exposing
    ``add_request(token_ids, num_computed, blocks)`` and ``remove_request(row)``
    (the CUDA library's or the oracle's); return {handle: row}."""
    rows = {}
    for op in wl.ops:
        if op[0] == "add":
            r = op[1]
            rows[r.handle] = state.add_request(r.token_ids, r.num_computed, r.blocks)
        else:
            state.remove_request(rows.pop(op[1]))
    return rows


def schedule_arrays(wl: Workload, rows: dict):
    """(rows[n], num_scheduled_tokens[n]) int32, in schedule-output order."""
    r = np.array([rows[h] for h, _ in wl.schedule], dtype=np.int32)
    ns = np.array([c for _, c in wl.schedule], dtype=np.int32)
    return r, ns


def group_tuples(wl: Workload):
    return [(g.block_size, g.max_blocks_per_req, g.num_blocks) for g in wl.groups]
