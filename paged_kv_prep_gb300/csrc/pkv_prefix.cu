// Prefix-cache block keys and the device index of cached blocks.
//
// "Prefix Cache" section of "从源码读 vLLM Scheduler": what is hashed is a
// token block together with its prefix context; the hash only indexes cached
// blocks, and a hit reuses the block's K/V; hits are limited to num_tokens - 1
// so the last position is always recomputed.  The page does not fix the hash.
// Reading: digest_j = FNV-1a 64 over the little-endian bytes of block j's token
// ids; key_j = key_{j-1} * P + digest_j (mod 2^64), key_{-1} = the FNV offset
// basis, P = the FNV prime.
//
// GB300 design.  Two passes.  The digests of all blocks are independent: the
// first pass spreads every block of every request evenly over the threads,
// one thread per block reading its tokens as 16-byte vectors through L1 when
// every block starts 16-byte aligned, else from a warp-private shared-memory
// row that the warp filled with coalesced 128-byte loads.  The chain is an
// affine recurrence, x -> P * x + d, and affine maps compose associatively,
// so the second pass turns each request's digests into keys: a warp per
// request of up to 256 blocks, a CTA per longer one; every lane folds a
// contiguous run into one map, the maps are scanned, and every lane replays
// its run.  The index is an open-addressing table of 64-bit keys in device
// memory (linear probing, atomicCAS inserts, bounded probes).  A match probes
// every key of the batch below its request's cap with a thread of its own and
// keeps each request's first miss (batches above PKV_MAX_BATCH requests: one
// CTA per request probing 256 keys per round, stopping at the first miss).
#include <string.h>

#include "pkv_async.cuh"
#include "pkv_common.cuh"

struct pkv_prefix_cache {
    int device = 0;
    int64_t capacity = 0;      // power of two
    unsigned long long *d_keys = nullptr;   // 0 = empty
    int32_t *d_ids = nullptr;
};

namespace {

using namespace pkv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kBasis = 0xcbf29ce484222325ULL;
constexpr uint64_t kPrime = 0x00000100000001b3ULL;
constexpr size_t kMaxKeysSmem = (PKV_MAX_BATCH + 1) * 4;   // the staged offsets

// composition of affine maps: first l, then r
struct Affine {
    uint64_t m, a;
};
__device__ __forceinline__ Affine compose(Affine l, Affine r) { return {l.m * r.m, l.a * r.m + r.a}; }

__device__ __forceinline__ Affine shfl_up(Affine v, int d) {
    return {__shfl_up_sync(0xffffffffu, v.m, d), __shfl_up_sync(0xffffffffu, v.a, d)};
}

// One FNV-1a byte step, h = (h ^ byte) * P mod 2^64, on the two 32-bit
// halves.  P = 2^40 + 0x1b3, so h * P = h * 0x1b3 + (h << 40): the low half
// is the low word of lo * 0x1b3, the high half gathers that product's high
// word, hi * 0x1b3 and lo << 8 (the part of h << 40 that stays below 2^64).
__device__ __forceinline__ void fnv_step(uint32_t &lo, uint32_t &hi, uint32_t byte) {
    constexpr uint32_t kPrimeLow = 0x1b3u;
    lo ^= byte;
    const uint32_t plo = lo * kPrimeLow;
    const uint32_t phi = __umulhi(lo, kPrimeLow);
    hi = hi * kPrimeLow + phi + (lo << 8);
    lo = plo;
}
static_assert(kPrime == (1ull << 40) + 0x1b3ull, "the FNV-1a 64 prime");

// Shared-memory row pitch of a warp's staged segments: 36 words, so every
// row starts 16-byte aligned and lane t reads its row as 16-byte vectors; the
// 8 lanes of a quarter-warp phase then hit banks 4 * (t + k) mod 32, all
// distinct -- no conflicts -- and a warp writing one row writes 32
// consecutive words.
constexpr int kSegTokens = 32;              // tokens of a block staged per round
constexpr int kPitch = kSegTokens + 4;

__device__ __forceinline__ int4 ld_vec(const int4 *p) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int32_t ld_token(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Pass 1: the FNV-1a digest of every block of every request.  Warps take
// tiles of 32 consecutive blocks in flat order (every warp gets the same work,
// whatever the mix of request lengths).  Lane t owns block t of the tile and
// finds its source row; then the warp stages the tile round by round, each
// round 32 tokens of every block: one load instruction per block, its 32 lanes
// reading 32 consecutive token ids (128 bytes, coalesced), all the round's
// loads in flight before the stores to shared memory.  After a warp-level
// sync each lane folds its own row into its digest.  No block-wide barrier.
// The digests go to keys[], where pass 2 turns them into chained keys.
__global__ void __launch_bounds__(kThreads) block_digest_kernel(
    const int32_t *rows, const int32_t *offsets, int32_t n, const int32_t *tokens,
    int64_t tok_stride, int32_t bs, int32_t total, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t smem[];
    int32_t *s_off = smem;                                   // [n + 1]
    __shared__ __align__(16) int32_t s_seg[kWarps][32 * kPitch];   // staged segments
    __shared__ const int32_t *s_src[kWarps][32];             // each block's first token
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int32_t e = tid; e <= n; e += kThreads) s_off[e] = offsets[e];
    __syncthreads();
    int32_t *seg = s_seg[warp];
    const int64_t tiles = (static_cast<int64_t>(total) + 31) / 32;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    // lane t's block of tile `tile`, its first token written to s_src[warp][t]
    auto locate = [&](int64_t tile) {
        const int64_t j = tile * 32 + lane;
        if (j < total) {
            // the request whose blocks contain j: last i with s_off[i] <= j
            int lo = 0, hi = n;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= j) lo = mid; else hi = mid;
            }
            s_src[warp][lane] = tokens + static_cast<int64_t>(rows[lo]) * tok_stride +
                                (j - s_off[lo]) * bs;
        }
        __syncwarp();
    };
    // one round of a tile: tokens [r0, r0 + len) of each of its nblk blocks,
    // one coalesced load instruction per block
    auto load_round = [&](int nblk, int32_t r0, int32_t len, int32_t (&v)[32]) {
#pragma unroll
        for (int q = 0; q < 32; q++)
            if (q < nblk && lane < len) v[q] = ld_token(s_src[warp][q] + r0 + lane);
    };
    int64_t tile = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    if (tile >= tiles) return;
    int32_t v[32];
    locate(tile);
    int nblk = static_cast<int>(total - tile * 32 < 32 ? total - tile * 32 : 32);
    load_round(nblk, 0, bs < kSegTokens ? bs : kSegTokens, v);
    for (;;) {
        const int64_t j = tile * 32 + lane;
        const bool mine = j < total;
        uint64_t h = kBasis;
        for (int32_t r0 = 0; r0 < bs; r0 += kSegTokens) {
            const int32_t len = bs - r0 < kSegTokens ? bs - r0 : kSegTokens;
#pragma unroll
            for (int q = 0; q < 32; q++)
                if (q < nblk && lane < len) seg[q * kPitch + lane] = v[q];
            __syncwarp();
            // the next round's loads go out before this round is hashed: the
            // rest of this tile, else the first round of the warp's next tile
            const int32_t r1 = r0 + kSegTokens;
            int64_t next_tile = tile;
            int next_nblk = nblk;
            if (r1 < bs) {
                load_round(nblk, r1, bs - r1 < kSegTokens ? bs - r1 : kSegTokens, v);
            } else if (tile + nwarps < tiles) {
                next_tile = tile + nwarps;
                next_nblk = static_cast<int>(total - next_tile * 32 < 32 ? total - next_tile * 32 : 32);
                // every lane has issued its loads from the old sources
                __syncwarp();
                locate(next_tile);
                load_round(next_nblk, 0, bs < kSegTokens ? bs : kSegTokens, v);
            }
            if (mine) {
                const int32_t *row = seg + lane * kPitch;
                uint32_t lo = static_cast<uint32_t>(h), hi = static_cast<uint32_t>(h >> 32);
                if (len == kSegTokens) {   // a full segment: 8 vector reads, unrolled
#pragma unroll
                    for (int k4 = 0; k4 < kSegTokens / 4; k4++) {
                        const int4 w = *reinterpret_cast<const int4 *>(row + 4 * k4);
                        const uint32_t ts[4] = {static_cast<uint32_t>(w.x), static_cast<uint32_t>(w.y),
                                                static_cast<uint32_t>(w.z), static_cast<uint32_t>(w.w)};
#pragma unroll
                        for (int e = 0; e < 4; e++)
#pragma unroll
                            for (int x = 0; x < 4; x++) fnv_step(lo, hi, (ts[e] >> (8 * x)) & 0xffu);
                    }
                } else {
                    for (int32_t k = 0; k < len; k++) {
                        const uint32_t t = static_cast<uint32_t>(row[k]);
#pragma unroll
                        for (int x = 0; x < 4; x++) fnv_step(lo, hi, (t >> (8 * x)) & 0xffu);
                    }
                }
                h = (static_cast<uint64_t>(hi) << 32) | lo;
            }
            __syncwarp();
            if (r1 >= bs) {
                if (mine) keys[j] = h;
                if (next_tile == tile) return;   // the warp's last tile
                tile = next_tile;
                nblk = next_nblk;
            }
        }
    }
}

// Pass 1 when every block's tokens start 16-byte aligned: thread j hashes
// block j straight from global memory, four tokens (one 16-byte vector) per
// load, through L1 (a warp's 32 blocks are mostly adjacent runs of token ids,
// so the loads of neighbouring lanes share cache lines); two vectors are in
// flight ahead of the one being hashed.
__global__ void __launch_bounds__(kThreads) block_digest_direct_kernel(
    const int32_t *rows, const int32_t *offsets, int32_t n, const int32_t *tokens,
    int64_t tok_stride, int32_t bs, int32_t total, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t smem[];
    int32_t *s_off = smem;                                   // [n + 1]
    for (int32_t e = threadIdx.x; e <= n; e += kThreads) s_off[e] = offsets[e];
    __syncthreads();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int nv = bs / 4;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < total;
         j += stride) {
        int lo = 0, hi = n;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= j) lo = mid; else hi = mid;
        }
        const int4 *src = reinterpret_cast<const int4 *>(
            tokens + static_cast<int64_t>(rows[lo]) * tok_stride + (j - s_off[lo]) * bs);
        uint32_t hl = static_cast<uint32_t>(kBasis), hh = static_cast<uint32_t>(kBasis >> 32);
        int4 w0 = ld_vec(src);
        int4 w1 = nv > 1 ? ld_vec(src + 1) : w0;
        for (int k = 0; k < nv; k++) {
            const int4 w2 = k + 2 < nv ? ld_vec(src + k + 2) : w1;
            const uint32_t ts[4] = {static_cast<uint32_t>(w0.x), static_cast<uint32_t>(w0.y),
                                    static_cast<uint32_t>(w0.z), static_cast<uint32_t>(w0.w)};
#pragma unroll
            for (int e = 0; e < 4; e++)
#pragma unroll
                for (int x = 0; x < 4; x++) fnv_step(hl, hh, (ts[e] >> (8 * x)) & 0xffu);
            w0 = w1;
            w1 = w2;
        }
        keys[j] = (static_cast<uint64_t>(hh) << 32) | hl;
    }
}

// Pass 2: each request's chain, key_j = key_{j-1} * P + digest_j (key_{-1} =
// the FNV offset basis), in place.  Two launches split the requests by length.
// Requests of up to kShortChain blocks: one warp each; lane l folds a
// contiguous run of at most 8 blocks into one affine map x -> m x + a, the
// warp scans the 32 maps with shuffles, and each lane replays its run from
// the key before it.  Longer requests: one CTA each, the same with 256 runs
// (at most ceil(blocks / 256) blocks, 16 for a 4096-block request) and a
// second level over the warps' totals.  A run of at most kRegRun digests is
// loaded into registers with all its loads in flight together and replayed
// from them (one trip to memory for the digests); a longer run is read in
// pieces of kRegRun, once to fold and again to replay.
constexpr int kRegRun = 16;

// i / run for 0 <= i < 2^16 and 1 <= run <= 16, by a multiply: with magic =
// ceil(2^32 / run) (run_magic), i * magic / 2^32 exceeds i / run by less than
// i * run / 2^32 < 2^-12, too little to cross the next integer.  run = 1 needs
// 2^32, which does not fit, and is taken apart.
__device__ __forceinline__ uint32_t run_magic(int32_t run) {
    return run > 1 ? 0xffffffffu / static_cast<uint32_t>(run) + 1u : 0u;
}
__device__ __forceinline__ int32_t div_run(int32_t i, int32_t run, uint32_t magic) {
    return run > 1 ? static_cast<int32_t>(__umulhi(static_cast<uint32_t>(i), magic)) : i;
}

// The digests of blocks [b0, b0 + n), n <= R, into registers.
template <int R>
__device__ __forceinline__ void load_run(uint64_t (&d)[R], const uint64_t *k, int32_t b0,
                                         int32_t n) {
#pragma unroll
    for (int u = 0; u < R; u++)
        if (u < n) d[u] = k[b0 + u];
}

// The map of a run held in registers (first block first).
template <int R>
__device__ __forceinline__ Affine fold_regs(const uint64_t (&d)[R], int32_t n) {
    Affine v = {1, 0};
#pragma unroll
    for (int u = 0; u < R; u++)
        if (u < n) v = compose(v, Affine{kPrime, d[u]});
    return v;
}

// Write the keys of the run held in registers, x being the key before it;
// returns the run's last key.
template <int R>
__device__ __forceinline__ uint64_t replay_regs(uint64_t x, const uint64_t (&d)[R], uint64_t *k,
                                                int32_t b0, int32_t n) {
#pragma unroll
    for (int u = 0; u < R; u++) {
        if (u < n) {
            x = x * kPrime + d[u];
            k[b0 + u] = x;
        }
    }
    return x;
}

// Inclusive scan of the lanes' maps; returns the map of the lanes before.
__device__ __forceinline__ Affine warp_scan_before(Affine &v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Affine o = shfl_up(v, d);
        if (lane >= d) v = compose(o, v);
    }
    Affine before = shfl_up(v, 1);
    if (lane == 0) before = {1, 0};
    return before;
}

constexpr int32_t kShortChain = 256;   // blocks a single warp chains
constexpr int kShortRun = kShortChain / 32;

__global__ void __launch_bounds__(kThreads, 4) chain_short_kernel(const int32_t *offsets,
                                                               int32_t n, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); r < n;
         r += nwarps) {
        const int32_t o0 = offsets[r];
        const int32_t nb = offsets[r + 1] - o0;
        if (nb > kShortChain) continue;   // chained by chain_long_kernel
        const int32_t run = (nb + 31) >> 5;   // at most kShortRun
        const int32_t b0 = min(nb, lane * run), b1 = min(nb, b0 + run);
        uint64_t *k = keys + o0;
        uint64_t d[kShortRun];
        load_run(d, k, b0, b1 - b0);
        Affine v = fold_regs(d, b1 - b0);
        const Affine before = warp_scan_before(v, lane);
        replay_regs(before.m * kBasis + before.a, d, k, b0, b1 - b0);
    }
}

// One CTA per entry of `spans`, the (first key, block count) of every
// request of more than kShortChain blocks, listed by the host, which knows
// every request's block count.  The list came with the call's one host copy,
// which the kernels before this one already waited for, so it is read before
// the wait for the digests.
__global__ void __launch_bounds__(kThreads, 4) chain_long_kernel(const int2 *spans, int32_t nlong,
                                                              uint64_t *keys) {
    int2 span = blockIdx.x < static_cast<unsigned>(nlong) ? spans[blockIdx.x] : make_int2(0, 0);
    pdl_wait();
    pdl_trigger();
    __shared__ Affine s_warp[kWarps];
    // a request of at most kThreads * kRegRun blocks passes through here:
    // thread t's run at row t (pitch kRegRun + 1: 8-byte rows 136 bytes apart,
    // at most two lanes of a warp on one bank pair)
    __shared__ uint64_t s_run[kThreads * (kRegRun + 1)];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = blockIdx.x; e < nlong; e += gridDim.x) {
        if (e != static_cast<int>(blockIdx.x)) span = spans[e];
        const int32_t o0 = span.x;
        const int32_t nb = span.y;
        const int32_t run = (nb + kThreads - 1) / kThreads;
        const int32_t b0 = min(nb, tid * run), b1 = min(nb, b0 + run);
        uint64_t *k = keys + o0;
        const bool staged = run <= kRegRun;   // the same for the whole CTA
        const uint32_t magic = run_magic(run);   // digest i belongs to thread i / run
        uint64_t d[kRegRun];
        Affine v = {1, 0};
        if (staged) {
            // coalesced loads of the request's digests, all in flight, into
            // the threads' rows
#pragma unroll
            for (int j = 0; j < kRegRun; j++) {
                const int32_t i = tid + j * kThreads;
                if (i < nb) d[j] = k[i];
            }
#pragma unroll
            for (int j = 0; j < kRegRun; j++) {
                const int32_t i = tid + j * kThreads;
                if (i < nb) {
                    const int32_t t = div_run(i, run, magic);
                    s_run[t * (kRegRun + 1) + (i - t * run)] = d[j];
                }
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < kRegRun; u++)
                if (u < b1 - b0) d[u] = s_run[tid * (kRegRun + 1) + u];
            v = fold_regs(d, b1 - b0);
        } else {
            // the run in pieces of kRegRun digests, read once to fold and
            // again to replay
            for (int32_t c = b0; c < b1; c += kRegRun) {
                const int32_t m = min(kRegRun, b1 - c);
                load_run(d, k, c, m);
                v = compose(v, fold_regs(d, m));
            }
        }
        Affine before = warp_scan_before(v, lane);   // this warp's runs before this one
        if (lane == 31) s_warp[warp] = v;
        __syncthreads();
        Affine lead = {1, 0};                        // the earlier warps' runs
        for (int w = 0; w < warp; w++) lead = compose(lead, s_warp[w]);
        before = compose(lead, before);
        uint64_t x = before.m * kBasis + before.a;
        if (staged) {
            // the keys back into the thread's row, then coalesced stores
#pragma unroll
            for (int u = 0; u < kRegRun; u++) {
                if (u < b1 - b0) {
                    x = x * kPrime + d[u];
                    s_run[tid * (kRegRun + 1) + u] = x;
                }
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kRegRun; j++) {
                const int32_t i = tid + j * kThreads;
                if (i < nb) {
                    const int32_t t = div_run(i, run, magic);
                    k[i] = s_run[t * (kRegRun + 1) + (i - t * run)];
                }
            }
        } else {
            for (int32_t c = b0; c < b1; c += kRegRun) {
                const int32_t m = min(kRegRun, b1 - c);
                load_run(d, k, c, m);
                x = replay_regs(x, d, k, c, m);
            }
        }
        __syncthreads();   // s_warp is rewritten for the next long request
    }
}

__global__ void __launch_bounds__(kThreads) insert_kernel(unsigned long long *table_keys,
                                                          int32_t *table_ids, int64_t mask,
                                                          const uint64_t *keys,
                                                          const int32_t *ids, int64_t count,
                                                          int32_t *err) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const unsigned long long key = keys[i];
        if (key == 0) continue;   // 0 marks an empty slot: such a block is never cached
        int64_t h = static_cast<int64_t>(key & static_cast<unsigned long long>(mask));
        bool placed = false;
        for (int64_t probe = 0; probe <= mask; probe++) {
            const unsigned long long old = atomicCAS(&table_keys[h], 0ull, key);
            if (old == 0ull) {
                table_ids[h] = ids[i];
                placed = true;
                break;
            }
            if (old == key) {   // already cached: the first id stays
                placed = true;
                break;
            }
            h = (h + 1) & mask;
        }
        if (!placed && err) atomicOr(err, PKV_DEVERR_TABLE_FULL);
    }
}

// One CTA per request: each round probes the next 256 keys in parallel and
// the request's hits end at the first uncached block.
__global__ void __launch_bounds__(kThreads) match_kernel(
    const unsigned long long *table_keys, const int32_t *table_ids, int64_t mask,
    const uint64_t *keys, const int32_t *offsets, const int32_t *max_hits, int32_t n,
    int32_t *hit_blocks, int32_t *hit_ids) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t s_first_miss;
    const int tid = threadIdx.x;
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t o0 = offsets[i];
        const int32_t nk = offsets[i + 1] - o0;
        const int32_t cap = min(nk, max(0, max_hits[i]));
        int32_t hits = cap;
        bool open = true;
        for (int32_t base = 0; base < nk; base += kThreads) {
            const int32_t j = base + tid;
            int32_t id = -1;
            bool found = false;
            if (open && j < cap) {
                const unsigned long long key = keys[o0 + j];
                if (key != 0) {
                    int64_t h = static_cast<int64_t>(key & static_cast<unsigned long long>(mask));
                    for (int64_t probe = 0; probe <= mask; probe++) {
                        const unsigned long long k = table_keys[h];
                        if (k == key) {
                            found = true;
                            id = table_ids[h];
                            break;
                        }
                        if (k == 0ull) break;
                        h = (h + 1) & mask;
                    }
                }
            }
            // the first key of this round (below the cap) that is not cached
            if (tid == 0) s_first_miss = kThreads;
            __syncthreads();
            if (open && j < cap && !found) atomicMin(&s_first_miss, tid);
            __syncthreads();
            const int first_miss = s_first_miss;
            if (j < nk) hit_ids[o0 + j] = (open && tid < first_miss && j < cap) ? id : -1;
            if (open && first_miss < kThreads) {
                hits = base + first_miss;
                open = false;
            }
            if (open && base + kThreads >= cap) open = false;   // everything up to the cap hit
            __syncthreads();
        }
        if (tid == 0) hit_blocks[i] = hits;
    }
}

// The flat match, for batches whose offsets fit in shared memory
// (n <= PKV_MAX_BATCH): every probe is independent, so the keys are spread
// evenly over the grid whatever the request lengths.
//   1. match_init_kernel: hit_blocks[i] = the request's cap;
//   2. match_probe_kernel: one lane per key below its request's cap probes the
//      index and writes its id (or -1); the lanes of a warp that belong to one
//      request (__match_any_sync) take the minimum of their misses and lower
//      hit_blocks[i] to it with one atomicMin; a key at or past a miss already
//      recorded is not probed;
//   3. match_mask_kernel: one warp per request writes -1 over the ids at and
//      past the request's first miss.
__global__ void __launch_bounds__(kThreads) match_init_kernel(const int32_t *offsets,
                                                              const int32_t *max_hits, int32_t n,
                                                              int32_t *hit_blocks) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int32_t nk = offsets[i + 1] - offsets[i];
        hit_blocks[i] = min(nk, max(0, max_hits[i]));
    }
}

__global__ void __launch_bounds__(kThreads) match_probe_kernel(
    const unsigned long long *table_keys, const int32_t *table_ids, int64_t mask,
    const uint64_t *keys, const int32_t *offsets, int32_t n, int32_t *hit_blocks,
    int32_t *hit_ids) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t s_off[];   // [n + 1]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int32_t e = tid; e <= n; e += kThreads) s_off[e] = offsets[e];
    __syncthreads();
    const int64_t total = s_off[n];
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t base = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * 32; base < total;
         base += nwarps * 32) {
        const int64_t j = base + lane;
        const bool valid = j < total;
        int32_t i = 0, jj = 0;
        bool miss = false;
        if (valid) {
            int lo = 0, hi = n;   // last i with s_off[i] <= j
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= j) lo = mid; else hi = mid;
            }
            i = lo;
            jj = static_cast<int32_t>(j - s_off[i]);
            // the cap, lowered by misses already recorded (a stale value only
            // costs a probe)
            const int32_t limit = *reinterpret_cast<volatile int32_t *>(&hit_blocks[i]);
            int32_t id = -1;
            if (jj < limit) {
                const unsigned long long key = keys[j];
                bool found = false;
                if (key != 0) {
                    int64_t h = static_cast<int64_t>(key & static_cast<unsigned long long>(mask));
                    for (int64_t probe = 0; probe <= mask; probe++) {
                        const unsigned long long k = table_keys[h];
                        if (k == key) {
                            found = true;
                            id = table_ids[h];
                            break;
                        }
                        if (k == 0ull) break;
                        h = (h + 1) & mask;
                    }
                }
                miss = !found;
            }
            hit_ids[j] = id;
        }
        // per request within the warp: the earliest miss, one atomic
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? i : -1 - lane);
        const int32_t first = static_cast<int32_t>(
            __reduce_min_sync(peers, static_cast<uint32_t>(miss ? jj : INT_MAX)));
        if (valid && first != INT_MAX && lane == __ffs(peers) - 1) atomicMin(&hit_blocks[i], first);
    }
}

__global__ void __launch_bounds__(kThreads) match_mask_kernel(const int32_t *offsets, int32_t n,
                                                              const int32_t *hit_blocks,
                                                              int32_t *hit_ids) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); i < n;
         i += nwarps) {
        const int32_t o0 = offsets[i];
        const int32_t nk = offsets[i + 1] - o0;
        for (int32_t jj = hit_blocks[i] + lane; jj < nk; jj += 32) hit_ids[o0 + jj] = -1;
    }
}

unsigned grid_for(int64_t items, int64_t per_block, int num_sms) {
    const int64_t need = (items + per_block - 1) / per_block;
    const int64_t wave = static_cast<int64_t>(num_sms) * (2048 / kThreads);
    return static_cast<unsigned>(need < 1 ? 1 : (need < wave ? need : wave));
}

int device_sms(int *out) {
    int dev = 0;
    PKV_CUDA_TRY(cudaGetDevice(&dev));
    PKV_CUDA_TRY(cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev));
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_block_keys(pkv_state *st, const int32_t *rows, int32_t n, int32_t block_size,
                   int32_t *out_offsets, uint64_t *d_keys, int64_t capacity, pkv_stream_t stream) {
    if (!st || !out_offsets || n < 0 || n > PKV_MAX_BATCH || block_size < 1)
        return PKV_ERR_INVALID_ARG;
    if (n > 0 && !rows) return PKV_ERR_INVALID_ARG;
    int64_t total = 0;
    out_offsets[0] = 0;
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        total += st->ntok[r] / block_size;
        if (total > INT32_MAX) return PKV_ERR_INVALID_ARG;
        out_offsets[i + 1] = static_cast<int32_t>(total);
    }
    if (!d_keys || total == 0) return PKV_OK;   // a size query, or nothing to hash
    if (capacity < total) return PKV_ERR_CAPACITY;
    // one host-to-device copy: rows, offsets at a 16-byte aligned offset, then
    // the (first key, block count) of the requests whose chain takes a whole
    // CTA (more than kShortChain blocks); at most 4 * (PKV_MAX_BATCH + 4)
    // words, the size of the state's staging array
    const int32_t n4 = (n + 3) & ~3;
    const int32_t o4 = (n + 1 + 3) & ~3;
    int status;
    char *buf = st->ring.reserve(static_cast<size_t>(n4 + o4 + 2 * n) * 4, &status);
    if (!buf) return status;
    memcpy(buf, rows, static_cast<size_t>(n) * 4);
    memcpy(buf + static_cast<size_t>(n4) * 4, out_offsets, static_cast<size_t>(n + 1) * 4);
    int32_t *spans = reinterpret_cast<int32_t *>(buf + static_cast<size_t>(n4 + o4) * 4);
    int32_t nlong = 0;
    for (int32_t i = 0; i < n; i++) {
        const int32_t nb = out_offsets[i + 1] - out_offsets[i];
        if (nb > kShortChain) {
            spans[2 * nlong] = out_offsets[i];
            spans[2 * nlong + 1] = nb;
            nlong++;
        }
    }
    cudaStream_t s = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(st->d_sched, buf,
                                    static_cast<size_t>(n4 + o4 + 2 * nlong) * 4,
                                    cudaMemcpyHostToDevice, s);
    const int rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    const size_t smem = static_cast<size_t>(n + 1) * 4;   // the offsets
    static int configured[64] = {0};
    if (st->device >= 0 && st->device < 64 && !configured[st->device]) {
        PKV_CUDA_TRY(cudaFuncSetAttribute(block_digest_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kMaxKeysSmem)));
        configured[st->device] = 1;
    }
    int per_sm = 0;
    PKV_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, block_digest_kernel,
                                                               kThreads, smem));
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = (total + kThreads - 1) / kThreads;   // 8 warp tiles each
    const int64_t wave = static_cast<int64_t>(st->num_sms) * per_sm;
    const unsigned grid1 = static_cast<unsigned>(tiles < wave ? tiles : wave);
    const int32_t *d_rows = st->d_sched;
    const int32_t *d_off = st->d_sched + n4;
    const bool direct = block_size % 4 == 0 && st->max_len % 4 == 0 &&
                        reinterpret_cast<uintptr_t>(st->d_tokens) % 16 == 0;
    if (direct) {
        static int configured_d[64] = {0};
        if (st->device >= 0 && st->device < 64 && !configured_d[st->device]) {
            PKV_CUDA_TRY(cudaFuncSetAttribute(block_digest_direct_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kMaxKeysSmem)));
            configured_d[st->device] = 1;
        }
        int per_sm_d = 0;
        PKV_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm_d, block_digest_direct_kernel, kThreads, smem));
        if (per_sm_d < 1) per_sm_d = 1;
        const int64_t ctas = (total + kThreads - 1) / kThreads;
        const int64_t wave_d = static_cast<int64_t>(st->num_sms) * per_sm_d;
        PKV_CUDA_TRY(launch_pdl(block_digest_direct_kernel,
                                dim3(static_cast<unsigned>(ctas < wave_d ? ctas : wave_d)),
                                dim3(kThreads), smem, s, d_rows, d_off, n,
                                static_cast<const int32_t *>(st->d_tokens),
                                static_cast<int64_t>(st->max_len), block_size,
                                static_cast<int32_t>(total), d_keys));
    } else {
        PKV_CUDA_TRY(launch_pdl(block_digest_kernel, dim3(grid1), dim3(kThreads), smem, s, d_rows,
                                d_off, n, static_cast<const int32_t *>(st->d_tokens),
                                static_cast<int64_t>(st->max_len), block_size,
                                static_cast<int32_t>(total), d_keys));
    }
    // the chains: short requests a warp each, long ones a CTA each
    const int64_t wave2 = static_cast<int64_t>(st->num_sms) * (2048 / kThreads);
    const int64_t ctas_short = (static_cast<int64_t>(n) + kWarps - 1) / kWarps;
    PKV_CUDA_TRY(launch_pdl(chain_short_kernel,
                            dim3(static_cast<unsigned>(ctas_short < wave2 ? ctas_short : wave2)),
                            dim3(kThreads), 0, s, d_off, n, d_keys));
    if (nlong > 0)
        PKV_CUDA_TRY(launch_pdl(chain_long_kernel, dim3(static_cast<unsigned>(nlong)),
                                dim3(kThreads), 0, s,
                                reinterpret_cast<const int2 *>(st->d_sched + n4 + o4), nlong,
                                d_keys));
    return PKV_OK;
}

int pkv_prefix_cache_create(pkv_prefix_cache **out, int64_t capacity, pkv_stream_t stream) {
    if (!out || capacity < 2 || (capacity & (capacity - 1)) || capacity > (int64_t(1) << 32))
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_prefix_cache *pc = new (std::nothrow) pkv_prefix_cache();
    if (!pc) return PKV_ERR_INVALID_ARG;
    pc->capacity = capacity;
    cudaError_t e = cudaGetDevice(&pc->device);
    if (e == cudaSuccess) e = cudaMalloc(&pc->d_keys, static_cast<size_t>(capacity) * 8);
    if (e == cudaSuccess) e = cudaMalloc(&pc->d_ids, static_cast<size_t>(capacity) * 4);
    cudaStream_t s = as_stream(stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(pc->d_keys, 0, static_cast<size_t>(capacity) * 8, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(pc->d_ids, 0xFF, static_cast<size_t>(capacity) * 4, s);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        cudaFree(pc->d_keys);
        cudaFree(pc->d_ids);
        delete pc;
        return PKV_ERR_CUDA;
    }
    *out = pc;
    return PKV_OK;
}

int pkv_prefix_cache_destroy(pkv_prefix_cache *pc) {
    if (!pc) return PKV_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(pc->d_keys);
    cudaFree(pc->d_ids);
    delete pc;
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

int pkv_prefix_cache_insert(pkv_prefix_cache *pc, const uint64_t *d_keys,
                            const int32_t *d_block_ids, int64_t count, int32_t *d_error,
                            pkv_stream_t stream) {
    if (!pc || count < 0 || (count > 0 && (!d_keys || !d_block_ids))) return PKV_ERR_INVALID_ARG;
    if (count == 0) return PKV_OK;
    int sms = 0;
    int rc = device_sms(&sms);
    if (rc != PKV_OK) return rc;
    PKV_CUDA_TRY(launch_pdl(insert_kernel, dim3(grid_for(count, kThreads, sms)), dim3(kThreads), 0,
                            as_stream(stream), pc->d_keys, pc->d_ids, pc->capacity - 1, d_keys,
                            d_block_ids, count, d_error));
    return PKV_OK;
}

int pkv_prefix_cache_match(pkv_prefix_cache *pc, const uint64_t *d_keys, const int32_t *d_offsets,
                           const int32_t *d_max_hits, int32_t n, int32_t *d_hit_blocks,
                           int32_t *d_hit_ids, pkv_stream_t stream) {
    if (!pc || n < 0) return PKV_ERR_INVALID_ARG;
    if (n == 0) return PKV_OK;
    if (!d_keys || !d_offsets || !d_max_hits || !d_hit_blocks || !d_hit_ids)
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    int rc = device_sms(&sms);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = as_stream(stream);
    if (n > PKV_MAX_BATCH) {   // offsets too many for shared memory: a CTA per request
        PKV_CUDA_TRY(launch_pdl(match_kernel, dim3(grid_for(n, 1, sms)), dim3(kThreads), 0, s,
                                pc->d_keys, pc->d_ids, pc->capacity - 1, d_keys, d_offsets,
                                d_max_hits, n, d_hit_blocks, d_hit_ids));
        return PKV_OK;
    }
    static int configured[64] = {0};
    if (pc->device >= 0 && pc->device < 64 && !configured[pc->device]) {
        PKV_CUDA_TRY(cudaFuncSetAttribute(match_probe_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>((PKV_MAX_BATCH + 1) * 4)));
        configured[pc->device] = 1;
    }
    const size_t smem = static_cast<size_t>(n + 1) * 4;
    int per_sm = 0;
    PKV_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, match_probe_kernel,
                                                               kThreads, smem));
    if (per_sm < 1) per_sm = 1;
    PKV_CUDA_TRY(launch_pdl(match_init_kernel, dim3(grid_for(n, kThreads, sms)), dim3(kThreads),
                            0, s, d_offsets, d_max_hits, n, d_hit_blocks));
    PKV_CUDA_TRY(launch_pdl(match_probe_kernel, dim3(static_cast<unsigned>(sms * per_sm)),
                            dim3(kThreads), smem, s, pc->d_keys, pc->d_ids, pc->capacity - 1,
                            d_keys, d_offsets, n, d_hit_blocks, d_hit_ids));
    PKV_CUDA_TRY(launch_pdl(match_mask_kernel, dim3(grid_for(n, kWarps, sms)), dim3(kThreads), 0,
                            s, d_offsets, n, static_cast<const int32_t *>(d_hit_blocks),
                            d_hit_ids));
    return PKV_OK;
}

}  // extern "C"
