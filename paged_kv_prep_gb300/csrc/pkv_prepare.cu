// Fused batch build: schedule output + request-state table -> flattened
// attention inputs, in one kernel launch.
//
// What it computes follows the page "Deep Dive into vLLM's Scheduling
// Mechanism: The Complete CPU-to-GPU Mapping Pipeline" (kongchang.com):
//   - "Extracting the Execution Batch from Global State": take the scheduled
//     requests, sort them by the number of tokens they run this step (ascending,
//     equal counts in schedule order), record index_mapping;
//   - "Contiguous Token Sequence Processing": query_start_loc (prefix sum),
//     positions, input_ids;
//   - "Complete Input Preparation for the Attention Module": seq_lens;
//   - "Multi-Layer Coordinate Conversion Pipeline" / "Address Calculation
//     Example": per KV-cache group, slot = block_table[row][pos / bs] * bs +
//     pos % bs, and the gathered block-table rows.
//
// GB300 design.  The work is integer gather/scatter bound by HBM, dominated
// by the block-table row gather (8 * n * W bytes).  Rather than a separate sort
// kernel, a scan kernel and an expansion kernel, one grid does everything:
//   * every CTA stages the n scheduled counts and rows in shared memory (a
//     bulk copy from device memory, or from the kernel's parameters for a
//     small host schedule), validates them and scans the counts in 32-request
//     tiles in schedule order;
//   * the whole step is one flat space of work units, request i owning
//     alpha + n_i consecutive units (alpha 4-, 16- or 32-byte chunks of its
//     block-table rows, then one unit per token); each CTA takes an equal contiguous slice
//     of that space, so the grid is balanced whatever the mix of decodes and
//     long prefill chunks, and is sized to the SM count;
//   * a CTA needs each of its requests' batch rank and query_start_loc, i.e.
//     the request's place in the stable sort and the sum of the counts that
//     precede it.  Only decodes precede a decode (nothing has fewer than one
//     token), so a decode's rank and start are both the number of decodes
//     before it in schedule order: a prefix count of the tiles' decode lane
//     masks.  Any other request is ranked by comparing its packed
//     (count, index) key with every key in shared memory and reducing --
//     no grid-wide barrier and no second kernel;
//   * the block-table rows move as 4-, 16- or 32-byte vectors, the first
//     round of loads issued before the ranks are known and several loads in
//     flight per thread before the stores; token units write positions,
//     input_ids and one int64 slot per group with coalesced accesses.
// Two narrower kernels give the same outputs where the general one would
// pay for structure the batch does not need (the host picks by shape):
// prepare_small_kernel for at most 32 requests with small tables (one CTA,
// the sort in one warp) and prepare_decode_kernel for pure decode steps
// (T == n: the sort is the identity, no ranks).
#include <limits.h>
#include <string.h>

#include <unordered_map>

#include "pkv_async.cuh"
#include "pkv_common.cuh"

namespace {

using namespace pkv;

constexpr int kThreads = 256;
constexpr int kBatch = 32;          // requests set up per round (one lane each of warps 0 and 1)
constexpr uint32_t kMaxPolls = 1u << 20;  // bounded mbarrier wait (~1 s at 1 us per poll)
constexpr int64_t kMinUnitsPerCta = 256;   // one unit per thread at least
// Schedules of up to this many requests from the host travel in the kernel's
// parameter block, which saves the host-to-device copy, its stream ordering
// and the kernel's read of the staged copy.  The block's size costs launch
// latency (about 0.6 us per KB), so there are kernels for a 32-request and a
// 256-request block, and the device-schedule path has none.
constexpr int kInlineMax = 256;
constexpr int kInlineSmall = 32;

struct PrepParams {
    const int32_t *rows;        // [n] request_state_index per scheduled request
    const int32_t *counts;      // [n] num_scheduled_tokens
    int32_t n;
    int32_t T;
    int32_t bulk_stage;         // counts and rows are 16-byte aligned: stage by bulk copy
    int32_t live_only;          // gather only the live block-table entries
    int32_t early;              // the schedule may be read before the previous kernel ends
    int32_t num_rows;
    int32_t max_len;
    int32_t G;
    int64_t tok_stride;
    const int32_t *completed;
    const int32_t *tokens;
    int64_t alpha;              // gather chunks per request (sum over groups)
    int64_t units_per_cta;
    int64_t total_units;
    int32_t chunk_off[PKV_MAX_GROUPS + 1];  // prefix over groups of units per row
    int32_t width[PKV_MAX_GROUPS];
    int32_t bs[PKV_MAX_GROUPS];
    int32_t bs_shift[PKV_MAX_GROUPS];       // log2(bs) when bs is a power of two, else -1
    int64_t num_blocks[PKV_MAX_GROUPS];
    const int32_t *table[PKV_MAX_GROUPS];
    int32_t *index_mapping;
    int32_t *qsl;
    int32_t *seq_lens;
    int32_t *positions;
    int32_t *input_ids;
    int32_t *out_table[PKV_MAX_GROUPS];
    int64_t *slots[PKV_MAX_GROUPS];
    int32_t *err;
    // device schedules: per-row claims of this call (rows listed twice), or null
    unsigned long long *stamp;
    uint32_t gen;
};

// The kernel's parameters: PrepParams, plus for NI > 0 a host schedule of at
// most NI requests (rows at [0, n), counts at [NI, NI + n)).
template <int NI>
struct PrepArgs {
    PrepParams p;
    int32_t sched[2 * NI];
};
template <>
struct PrepArgs<0> {
    PrepParams p;
};

__device__ __forceinline__ int4 ld_stream(const int4 *p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int32_t ld_stream(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void flag(int32_t *err, int32_t bit) {
    if (err) atomicOr(err, bit);
}

// One batch row per request ("Extracting the Execution Batch from Global
// State").  For a device schedule, request i of call `gen` claims its row's
// stamp (gen << 32 | i): it reads the stamp, and if that holds an older
// call, swaps in its own value.  A claim of the current call is never
// replaced, so every CTA that touches request i gets the same answer: the
// row is i's when the stamp read already holds i, when the swap succeeded,
// or when the swap lost to another CTA of request i.  (A swap can only lose
// to a claim of the current call.)
__device__ __forceinline__ unsigned long long stamp_of(uint32_t gen, int i) {
    return (static_cast<unsigned long long>(gen) << 32) | static_cast<uint32_t>(i);
}
__device__ __forceinline__ bool owns_row(unsigned long long seen, unsigned long long swap_result,
                                         bool swapped, uint32_t gen, int i) {
    const unsigned long long v = swapped && swap_result != seen ? swap_result : seen;
    if (swapped && swap_result == seen) return true;
    return (v >> 32) == gen && static_cast<uint32_t>(v) == static_cast<uint32_t>(i);
}

// A block-table chunk moved by one thread: 4, 16 or 32 bytes.
template <int CH>
struct Chunk;
template <>
struct Chunk<4> {
    int32_t v;
};
template <>
struct Chunk<16> {
    int4 v;
};
template <>
struct Chunk<32> {
    int4 a, b;
};

__device__ __forceinline__ void ld_chunk(Chunk<4> &c, const char *p) {
    c.v = ld_stream(reinterpret_cast<const int32_t *>(p));
}
__device__ __forceinline__ void ld_chunk(Chunk<16> &c, const char *p) {
    c.v = ld_stream(reinterpret_cast<const int4 *>(p));
}
__device__ __forceinline__ void ld_chunk(Chunk<32> &c, const char *p) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(c.a.x), "=r"(c.a.y), "=r"(c.a.z), "=r"(c.a.w), "=r"(c.b.x),
                   "=r"(c.b.y), "=r"(c.b.z), "=r"(c.b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st_chunk(char *p, const Chunk<4> &c) {
    *reinterpret_cast<int32_t *>(p) = c.v;
}
__device__ __forceinline__ void st_chunk(char *p, const Chunk<16> &c) {
    *reinterpret_cast<int4 *>(p) = c.v;
}
__device__ __forceinline__ void st_chunk(char *p, const Chunk<32> &c) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(c.a.x),
                 "r"(c.a.y), "r"(c.a.z), "r"(c.a.w), "r"(c.b.x), "r"(c.b.y), "r"(c.b.z),
                 "r"(c.b.w)
                 : "memory");
}
__device__ __forceinline__ void fill_null(Chunk<4> &c) { c.v = -1; }
__device__ __forceinline__ void fill_null(Chunk<16> &c) { c.v = make_int4(-1, -1, -1, -1); }
__device__ __forceinline__ void fill_null(Chunk<32> &c) {
    c.a = make_int4(-1, -1, -1, -1);
    c.b = c.a;
}

// Shared-memory layout of the staged schedule, in int32 words: the counts
// (later the packed rank keys), the rows, the 32-request tile sums, the
// decodes (count 1) per tile, and the tiles' decode lane masks.
struct SmemLayout {
    int n4, nt, rows, tile, ones, mask1, words;
};
__host__ __device__ inline SmemLayout smem_layout(int n) {
    SmemLayout l;
    l.n4 = (n + 3) & ~3;
    l.nt = (n + 31) / 32;
    l.rows = l.n4;
    l.tile = 2 * l.n4;                 // [nt + 1]
    l.ones = l.tile + l.nt + 1;        // [nt]
    l.mask1 = l.ones + l.nt;           // [nt]
    l.words = l.mask1 + l.nt;
    return l;
}

// Cooperative rank of up to W listed requests of a batch against a key array:
// each thread takes a slice of the keys, counts the keys that precede each
// request in (count, schedule index) order and sums their counts, then the
// partial results are reduced per warp and added into s_rank / s_start.
// Packed keys (count << 14 | index) make "precedes" one integer compare; with
// raw counts the key array is the whole schedule and ties compare indexes.
template <int W>
__device__ __forceinline__ void rank_slice(const int32_t *s_key, int len4, bool packed,
                                           const int32_t *s_cnt, int ib, const int32_t *s_list,
                                           int q0, int nlist, int32_t *s_rank,
                                           int32_t *s_start) {
    const int tid = threadIdx.x, lane = tid & 31;
    int32_t kq[W], cnt[W], sum[W];
#pragma unroll
    for (int u = 0; u < W; u++) {
        // INT_MIN: nothing precedes it
        kq[u] = q0 + u < nlist ? s_cnt[ib + s_list[q0 + u]] : INT_MIN;
        cnt[u] = 0;
        sum[u] = 0;
    }
    const int4 *k4 = reinterpret_cast<const int4 *>(s_key);
    for (int v = tid; v < len4 / 4; v += kThreads) {
        const int4 k = k4[v];
        const int32_t e[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
        for (int x = 0; x < 4; x++) {
            if (packed) {
                const int32_t c = e[x] >> 14;
#pragma unroll
                for (int u = 0; u < W; u++)
                    if (e[x] < kq[u]) {
                        cnt[u]++;
                        sum[u] += c;
                    }
            } else {
                const int j = 4 * v + x;
#pragma unroll
                for (int u = 0; u < W; u++)
                    if (e[x] < kq[u] ||
                        (e[x] == kq[u] && q0 + u < nlist && j < ib + s_list[q0 + u])) {
                        cnt[u]++;
                        sum[u] += e[x];
                    }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < W; u++) {
        if (q0 + u >= nlist) break;
        const int32_t c = __reduce_add_sync(0xffffffffu, cnt[u]);
        const int32_t sm = __reduce_add_sync(0xffffffffu, sum[u]);
        if (lane == 0) {
            const int q = s_list[q0 + u];
            atomicAdd(&s_rank[q], c);
            atomicAdd(&s_start[q], sm);
        }
    }
}

template <int CH, int NI>
__global__ void __launch_bounds__(kThreads, 3) prepare_kernel(const PrepArgs<NI> args) {
    const PrepParams &p = args.p;
    constexpr int kRound = 128 / CH > 8 ? 8 : 128 / CH;   // chunks in flight per thread
    extern __shared__ __align__(16) int32_t smem[];
    const int n = p.n;
    const SmemLayout L = smem_layout(n);
    const int n4 = L.n4;
    int32_t *s_cnt = smem;             // [n4] counts, later packed rank keys (padding INT_MAX)
    int32_t *s_rows = smem + L.rows;   // [n4] rows
    int32_t *s_tile = smem + L.tile;   // [nt + 1] tile sums, then their exclusive prefix
    int32_t *s_ones = smem + L.ones;   // [nt] decodes per tile, then their exclusive prefix
    uint32_t *s_mask1 = reinterpret_cast<uint32_t *>(smem + L.mask1);  // [nt] decode lanes

    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int64_t s_C[kBatch + 1];
    __shared__ int32_t s_rank[kBatch], s_start[kBatch], s_row[kBatch], s_comp[kBatch];
    __shared__ int32_t s_cnt_b[kBatch], s_ok[kBatch];
    __shared__ int32_t s_ga[kBatch], s_gpre[kBatch + 1], s_ka[kBatch], s_tpre[kBatch + 1];
    __shared__ const char *s_src[kBatch * PKV_MAX_GROUPS];
    __shared__ int32_t s_live[kBatch * PKV_MAX_GROUPS];
    // PKV_LIVE_TABLES: per (request, group), the first wanted chunk in the
    // slice and the wanted chunks of the request's earlier groups
    __shared__ int32_t s_wa[kBatch * PKV_MAX_GROUPS], s_wcum[kBatch * PKV_MAX_GROUPS];
    __shared__ char *s_dst[kBatch * PKV_MAX_GROUPS];
    __shared__ int32_t s_list[kBatch];   // batch positions ranked by comparison
    __shared__ int32_t s_nreq, s_more, s_flag, s_ib, s_nlist;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.G;

    // the state and the output buffers may be in use by the kernel launched
    // before this one, and so may the schedule unless it is known not to be
    // (in the parameters, copied in by a copy, or flagged settled): steps 1-3
    // read nothing else, so then the wait comes before step 4
    if (!p.early) pdl_wait();
    pdl_trigger();

    // ---- 1. stage the counts and the rows (bulk-copy engine) -----------------
    const int n_bulk = NI == 0 && p.bulk_stage ? (n & ~3) : 0;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0 && n_bulk > 0) {
        mbar_arrive_expect_tx(&s_bar, static_cast<uint32_t>(2 * n_bulk * 4));
        bulk_g2s(s_cnt, p.counts, static_cast<uint32_t>(n_bulk * 4), &s_bar);
        bulk_g2s(s_rows, p.rows, static_cast<uint32_t>(n_bulk * 4), &s_bar);
    }
    if constexpr (NI > 0) {
        for (int j = tid; j < n4; j += kThreads) {
            s_cnt[j] = j < n ? args.sched[NI + j] : INT_MAX;
            s_rows[j] = j < n ? args.sched[j] : 0;
        }
    } else {
        for (int j = n_bulk + tid; j < n4; j += kThreads) {
            s_cnt[j] = j < n ? ld_stream(p.counts + j) : INT_MAX;
            s_rows[j] = j < n ? ld_stream(p.rows + j) : 0;
        }
    }
    if (n_bulk > 0) {
        const bool arrived = __syncthreads_and(mbar_wait(&s_bar, 0, kMaxPolls));
        if (!arrived) {
            // give the copies one more bounded wait so none lands after exit
            if (tid == 0) flag(p.err, PKV_DEVERR_TIMEOUT);
            mbar_wait(&s_bar, 0, kMaxPolls);
            return;
        }
    }
    __syncthreads();

    // ---- 2. validate; 32-request tile sums; the decodes of each tile as a
    //         lane mask; packed rank keys.  A lane takes four consecutive
    //         counts (one 16-byte vector), so a warp covers four tiles per
    //         iteration.  The counts become packed keys in place (the raw
    //         counts are read again below if one of them does not fit)
    const int nt = L.nt;
    const int nvec = n4 / 4;
    int bad = 0, big = 0;
    for (int v0 = 32 * warp; v0 < nvec; v0 += kThreads) {
        const int v = v0 + lane;
        const int j0 = 4 * v;
        int4 c4 = make_int4(0, 0, 0, 0);
        if (v < nvec) c4 = reinterpret_cast<const int4 *>(s_cnt)[v];
        int32_t c[4] = {c4.x, c4.y, c4.z, c4.w};
        int32_t sum = 0;
        uint32_t nib = 0;
#pragma unroll
        for (int x = 0; x < 4; x++) {
            const bool valid = j0 + x < n;
            bad |= valid & ((c[x] < 1) | (c[x] > p.T));
            big |= valid & (c[x] > 65535);
            // counts are <= T < 2^26 unless flagged, so a tile sum fits in int32
            sum += valid ? c[x] : 0;
            nib |= static_cast<uint32_t>(valid && c[x] == 1) << x;
        }
        // the eight lanes of a tile: its sum and its decode lane mask
        uint32_t m = nib << (4 * (lane & 7));
#pragma unroll
        for (int d = 1; d < 8; d <<= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, d);
            m |= __shfl_xor_sync(0xffffffffu, m, d);
        }
        const int t = v >> 3;
        if ((lane & 7) == 0 && t < nt) {
            s_tile[t] = sum;
            s_mask1[t] = m;
            s_ones[t] = __popc(m);
        }
        // (count << 14 | index) < 2^30 orders requests exactly as (count,
        // index) when every count is <= 65535 (see `packed`)
#pragma unroll
        for (int x = 0; x < 4; x++)
            if (j0 + x < n)
                c[x] = static_cast<int32_t>((static_cast<uint32_t>(c[x]) << 14) |
                                            static_cast<uint32_t>(j0 + x));
        if (v < nvec) reinterpret_cast<int4 *>(s_cnt)[v] = make_int4(c[0], c[1], c[2], c[3]);
    }
    bad = __syncthreads_or(bad);
    const bool packed = !__syncthreads_or(big) && n <= 16384;
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) flag(p.err, PKV_DEVERR_COUNT);
        return;
    }
    // a count above 65535: rank by raw counts, read again from the schedule
    // (ordered before their first use by the barrier after the tile scan)
    if (!packed)
        for (int j = tid; j < n; j += kThreads)
            if constexpr (NI > 0) s_cnt[j] = args.sched[NI + j];
            else s_cnt[j] = ld_stream(p.counts + j);
    // exclusive prefix over the tiles (warp 0), in place; s_tile[nt] = total
    if (warp == 0) {
        int64_t carry = 0;
        int32_t carry1 = 0;
        for (int t0 = 0; t0 < nt; t0 += 32) {
            const int t = t0 + lane;
            // exact in 64 bits: a schedule whose true total differs from T
            // must not pass the check below by wrapping around
            const int64_t v = t < nt ? s_tile[t] : 0;
            const int32_t o = t < nt ? s_ones[t] : 0;
            int64_t inc = v;
            int32_t inc1 = o;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t x = __shfl_up_sync(0xffffffffu, inc, d);
                const int32_t x1 = __shfl_up_sync(0xffffffffu, inc1, d);
                if (lane >= d) {
                    inc += x;
                    inc1 += x1;
                }
            }
            if (t < nt) {
                s_tile[t] = static_cast<int32_t>(carry + inc - v);
                s_ones[t] = carry1 + inc1 - o;
            }
            carry += __shfl_sync(0xffffffffu, inc, 31);
            carry1 += __shfl_sync(0xffffffffu, inc1, 31);
        }
        if (lane == 0) {
            s_tile[nt] = static_cast<int32_t>(carry);
            s_flag = carry != p.T;
        }
    }
    __syncthreads();
    if (s_flag) {
        if (blockIdx.x == 0 && tid == 0) flag(p.err, PKV_DEVERR_COUNT);
        return;
    }
    // from here every prefix is <= T < 2^31
    auto count_of = [&](int i) -> int32_t { return packed ? (s_cnt[i] >> 14) : s_cnt[i]; };

    // ---- 3. this CTA's slice of the unit space -------------------------------
    // request i owns units [C(i), C(i+1)), C(i) = alpha * i + (sum of counts
    // before i in schedule order)
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * p.units_per_cta;
    const int64_t hi = min(lo + p.units_per_cta, p.total_units);
    if (lo >= hi) return;
    // last tile whose first request starts at or before lo
    int tl = 0, tr = nt;
    while (tr - tl > 1) {
        const int m = (tl + tr) >> 1;
        if (p.alpha * 32 * m + s_tile[m] <= lo) tl = m; else tr = m;
    }
    // warps 0 and 1 both carry the schedule-order prefix from batch to batch
    int ib = 0;
    int32_t carry = 0;
    if (warp < 2) {
        const int i = 32 * tl + lane;
        const int32_t c = i < n ? count_of(i) : 0;
        int32_t inc = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += o;
        }
        const int64_t Ci = p.alpha * i + s_tile[tl] + (inc - c);
        const unsigned le = __ballot_sync(0xffffffffu, i < n && Ci <= lo);
        const int first = 31 - __clz(le);            // lane 0 always qualifies
        ib = 32 * tl + first;
        carry = s_tile[tl] + __shfl_sync(0xffffffffu, inc - c, first);
    }

    // from here on the state is read and the outputs are written
    if (p.early) pdl_wait();

    for (;;) {
        // ---- 4. the batch's requests, one lane each: warp 0 lays out their
        //         chunk and token ranges, warp 1 reads their rows and sets up
        //         table pointers and initial ranks (two chains side by side)
        int32_t comp = 0;
        // warp 1, device schedules: the request's claim on its row (stamp read,
        // swap result), resolved after the ranks
        unsigned long long claim_seen = 0, claim_got = 0;
        bool claim_on = false, claim_swapped = false;
        if (warp < 2) {
            const int q = lane;
            const int i = ib + q;
            const int32_t cnt = i < n ? count_of(i) : 0;
            int32_t inc = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += o;
            }
            const int64_t c0 = p.alpha * i + carry + (inc - cnt);
            const bool in = i < n && c0 < hi;
            const unsigned in_mask = __ballot_sync(0xffffffffu, in);
            const int nreq = __popc(in_mask);
            if (warp == 0) {
                int32_t gcount = 0, tcount = 0;
                if (in) {
                    s_C[q] = c0;
                    const int64_t g_lo = max(lo, c0) - c0, g_hi = min(hi, c0 + p.alpha) - c0;
                    s_ga[q] = static_cast<int32_t>(g_lo);
                    gcount = g_hi > g_lo ? static_cast<int32_t>(g_hi - g_lo) : 0;
                    const int64_t t0 = c0 + p.alpha;
                    const int64_t k_lo = max(lo, t0) - t0, k_hi = min(hi, t0 + cnt) - t0;
                    s_ka[q] = static_cast<int32_t>(k_lo > 0 ? k_lo : 0);
                    tcount = k_hi > k_lo ? static_cast<int32_t>(k_hi - k_lo) : 0;
                }
                // inclusive scans of the per-request chunk and token counts
                int32_t gi = gcount, ti = tcount;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int32_t go = __shfl_up_sync(0xffffffffu, gi, d);
                    const int32_t to = __shfl_up_sync(0xffffffffu, ti, d);
                    if (lane >= d) {
                        gi += go;
                        ti += to;
                    }
                }
                if (in) {
                    // (with PKV_LIVE_TABLES warp 1 counts only the wanted chunks)
                    if (!p.live_only) s_gpre[q + 1] = gi;
                    s_tpre[q + 1] = ti;
                }
            } else {
                int32_t wcount = 0;
                if (in) {
                    const int32_t row = s_rows[i];
                    const bool in_table = row >= 0 && row < p.num_rows;
                    const bool ok = in_table;
                    // the claim is read here, next to completed_tokens, swapped
                    // before the rank loop and resolved after it (the stores
                    // are the first to need it)
                    claim_on = ok && p.stamp;
                    if (claim_on) claim_seen = __ldcg(p.stamp + row);
                    s_row[q] = row;
                    s_ok[q] = ok;
                    s_cnt_b[q] = cnt;
                    // a decode's rank and start are the decodes before it in
                    // schedule order (nothing else precedes a count of 1);
                    // every other request is ranked by comparison
                    int32_t r0 = 0;
                    if (packed && cnt == 1)
                        r0 = s_ones[i >> 5] + __popc(s_mask1[i >> 5] & ((1u << (i & 31)) - 1u));
                    s_rank[q] = r0;
                    s_start[q] = r0;
                    if (ok) comp = p.completed[row];   // consumed after the rank loop
                    else if (!in_table) flag(p.err, PKV_DEVERR_ROW);
                    for (int g = 0; g < G; g++) {
                        s_src[q * G + g] = ok ? reinterpret_cast<const char *>(
                                                    p.table[g] + static_cast<int64_t>(row) * p.width[g])
                                              : nullptr;
                        // live entries: the blocks of positions [0, completed + n)
                        int32_t live = p.width[g];
                        if (p.live_only) {
                            const int64_t len = static_cast<int64_t>(comp) + cnt;
                            const int64_t nb = (len + p.bs[g] - 1) / p.bs[g];
                            live = static_cast<int32_t>(nb < p.width[g] ? nb : p.width[g]);
                        }
                        s_live[q * G + g] = live;
                    }
                    if (p.live_only) {
                        // the wanted chunks of each group inside the slice: a
                        // chunk is wanted when it starts below the live entries
                        const int64_t g_lo = max(lo, c0) - c0, g_hi = min(hi, c0 + p.alpha) - c0;
                        int32_t cum = 0;
                        for (int g = 0; g < G; g++) {
                            const int64_t wg = (static_cast<int64_t>(s_live[q * G + g]) * 4 + CH - 1) / CH;
                            const int64_t a = max(g_lo, static_cast<int64_t>(p.chunk_off[g]));
                            const int64_t b = min(g_hi, static_cast<int64_t>(p.chunk_off[g]) + wg);
                            s_wa[q * G + g] = static_cast<int32_t>(a);
                            s_wcum[q * G + g] = cum;
                            cum += b > a ? static_cast<int32_t>(b - a) : 0;
                        }
                        wcount = cum;
                    }
                }
                if (p.live_only) {
                    int32_t wi = wcount;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const int32_t wo = __shfl_up_sync(0xffffffffu, wi, d);
                        if (lane >= d) wi += wo;
                    }
                    if (in) s_gpre[q + 1] = wi;
                }
                if (claim_on && (claim_seen >> 32) != p.gen) {
                    claim_got = atomicCAS(p.stamp + s_row[q], claim_seen, stamp_of(p.gen, i));
                    claim_swapped = true;
                }
                const bool cmp = in && !(packed && cnt == 1);
                const unsigned cmask = __ballot_sync(0xffffffffu, cmp);
                if (cmp) s_list[__popc(cmask & ((1u << lane) - 1u))] = q;
                if (lane == 0) s_nlist = __popc(cmask);
            }
            // the next batch starts after this one if the slice goes on
            carry += __shfl_sync(0xffffffffu, inc, nreq - 1);
            if (warp == 0 && lane == 0) {
                s_gpre[0] = 0;
                s_tpre[0] = 0;
                s_nreq = nreq;
                s_more = nreq == 32 && ib + 32 < n && p.alpha * (ib + 32) + carry < hi;
                s_ib = ib;
            }
        }
        __syncthreads();
        const int nreq = s_nreq;
        const int ibatch = s_ib;

        // locate flat gather chunk f: request qg (monotone per thread), group
        // g, byte offset within the group's row.  With PKV_LIVE_TABLES the
        // flat space holds only the wanted chunks (those that start below the
        // live entries); the others stay put.
        const int32_t gtotal = s_gpre[nreq];
        int qg = 0;
        auto locate_all = [&](int32_t f, int &g, int64_t &off) {
            while (qg + 1 < nreq && s_gpre[qg + 1] <= f) qg++;
            const int32_t chunk = s_ga[qg] + (f - s_gpre[qg]);
            g = 0;
            while (chunk >= p.chunk_off[g + 1]) g++;
            off = static_cast<int64_t>(chunk - p.chunk_off[g]) * CH;
        };
        auto locate_live = [&](int32_t f, int &g, int64_t &off) {
            while (qg + 1 < nreq && s_gpre[qg + 1] <= f) qg++;
            const int32_t k = f - s_gpre[qg];
            g = 0;
            while (g + 1 < G && k >= s_wcum[qg * G + g + 1]) g++;
            const int32_t chunk = s_wa[qg * G + g] + (k - s_wcum[qg * G + g]);
            off = static_cast<int64_t>(chunk - p.chunk_off[g]) * CH;
        };

        // ---- 5. first gather round in flight before the ranks are known -------
        Chunk<CH> v[kRound];
        // (each gather loop is written once and instantiated per mode, so the
        // mode is not tested per chunk)
        auto first_round = [&](auto locate) {
#pragma unroll
            for (int u = 0; u < kRound; u++) {
                const int32_t f = u * kThreads + tid;
                if (f < gtotal) {
                    int g;
                    int64_t off;
                    locate(f, g, off);
                    const char *src = s_src[qg * G + g];
                    if (src) ld_chunk(v[u], src + off); else fill_null(v[u]);
                }
            }
        };
        if (p.live_only) first_round(locate_live); else first_round(locate_all);

        // ---- 6. rank + query_start_loc of every request in the batch ---------
        // rank = #{j : (n_j, j) < (n_i, i)}, start = the sum of those n_j;
        // decodes are done, the listed requests count the keys below theirs
        const int nlist = s_nlist;
        const int32_t *keys = s_cnt;
        const int len4 = n4;
        for (int q0 = 0; q0 < nlist;) {
            const int left = nlist - q0;
            if (left >= 4) {
                rank_slice<4>(keys, len4, packed, s_cnt, ibatch, s_list, q0, nlist, s_rank, s_start);
                q0 += 4;
            } else if (left >= 2) {
                rank_slice<2>(keys, len4, packed, s_cnt, ibatch, s_list, q0, nlist, s_rank, s_start);
                q0 += 2;
            } else {
                rank_slice<1>(keys, len4, packed, s_cnt, ibatch, s_list, q0, nlist, s_rank, s_start);
                q0 += 1;
            }
        }
        if (warp == 1 && lane < nreq) {
            s_comp[lane] = comp;
            if (claim_on && !owns_row(claim_seen, claim_got, claim_swapped, p.gen, ib + lane)) {
                // another listing keeps the row: every output of this one is -1
                s_ok[lane] = 0;
                for (int g = 0; g < G; g++) s_src[lane * G + g] = nullptr;
                flag(p.err, PKV_DEVERR_DUP);
            }
        }
        __syncthreads();

        // ---- 7. per-request scalars (by the CTA owning the request's first
        //         unit) and the destination rows ------------------------------
        if (tid < nreq) {
            const int32_t rank = s_rank[tid];
            for (int g = 0; g < G; g++)
                s_dst[tid * G + g] = reinterpret_cast<char *>(
                    p.out_table[g] + static_cast<int64_t>(rank) * p.width[g]);
            if (s_C[tid] >= lo) {
                const bool ok = s_ok[tid];
                p.index_mapping[rank] = ok ? s_row[tid] : -1;
                p.qsl[rank] = s_start[tid];
                p.seq_lens[rank] = ok ? s_comp[tid] + s_cnt_b[tid] : -1;
                if (rank == n - 1) p.qsl[n] = s_start[tid] + s_cnt_b[tid];
            }
        }
        __syncthreads();

        // ---- 8. block-table row gather --------------------------------------
        auto gather_rest = [&](auto locate) {
            qg = 0;
#pragma unroll
            for (int u = 0; u < kRound; u++) {
                const int32_t f = u * kThreads + tid;
                if (f < gtotal) {
                    int g;
                    int64_t off;
                    locate(f, g, off);
                    if (!s_ok[qg]) fill_null(v[u]);   // loaded before its row was found repeated
                    st_chunk(s_dst[qg * G + g] + off, v[u]);
                }
            }
            for (int32_t f0 = kRound * kThreads; f0 < gtotal; f0 += kRound * kThreads) {
                char *dst[kRound];
#pragma unroll
                for (int u = 0; u < kRound; u++) {
                    const int32_t f = f0 + u * kThreads + tid;
                    dst[u] = nullptr;
                    if (f < gtotal) {
                        int g;
                        int64_t off;
                        locate(f, g, off);
                        const char *src = s_src[qg * G + g];
                        if (src) ld_chunk(v[u], src + off); else fill_null(v[u]);
                        dst[u] = s_dst[qg * G + g] + off;
                    }
                }
#pragma unroll
                for (int u = 0; u < kRound; u++)
                    if (dst[u]) st_chunk(dst[u], v[u]);
            }
        };
        if (p.live_only) gather_rest(locate_live); else gather_rest(locate_all);

        // ---- 9. per-token expansion ------------------------------------------
        const int32_t ttotal = s_tpre[nreq];
        int qt = 0;
        for (int32_t f = tid; f < ttotal; f += kThreads) {
            while (qt + 1 < nreq && s_tpre[qt + 1] <= f) qt++;
            const int32_t k = s_ka[qt] + (f - s_tpre[qt]);
            const int32_t t = s_start[qt] + k;
            const int32_t pos = s_comp[qt] + k;
            const int32_t row = s_row[qt];
            bool ok = s_ok[qt];
            if (ok && pos >= p.max_len) {
                flag(p.err, PKV_DEVERR_POSITION);
                ok = false;
            }
            const int32_t id = ok ? ld_stream(p.tokens + row * p.tok_stride + pos) : -1;
            for (int g = 0; g < G; g++) {
                int64_t slot = -1;
                if (ok) {
                    const int32_t bsz = p.bs[g];
                    const int32_t sh = p.bs_shift[g];
                    const int32_t lb = sh >= 0 ? (pos >> sh) : pos / bsz;
                    const int32_t off = pos - lb * bsz;
                    int32_t pb = -1;
                    if (lb < p.width[g]) pb = p.table[g][static_cast<int64_t>(row) * p.width[g] + lb];
                    if (pb >= 0 && pb < p.num_blocks[g])
                        slot = static_cast<int64_t>(pb) * bsz + off;
                    else
                        flag(p.err, PKV_DEVERR_BLOCK);
                }
                p.slots[g][t] = slot;
            }
            p.positions[t] = ok ? pos : -1;
            p.input_ids[t] = id;
        }
        const bool more = s_more;
        __syncthreads();
        if (!more) break;
        ib += 32;   // (used by warps 0 and 1, whose carry already covers this batch)
    }
}

// ---------------------------------------------------------------------------
// Small batches: at most 32 requests, at most 2048 tokens and 16384 table
// entries.  One CTA; the sort is one warp (lane i holds request i and counts
// the requests before it through shuffles), so there is no tile scan, slice
// search or staging, and a row listed twice in a device schedule is found in
// the same loop (the first listing keeps it).  What remains is about three
// dependent trips to memory: completed_tokens and the table rows (issued
// together: the full rows do not need it), then the token ids and the
// slots' block-table lookups.
// ---------------------------------------------------------------------------
constexpr int kSmallN = 32;
constexpr int32_t kSmallT = 2048;
constexpr int64_t kSmallEntries = 16384;

template <int NI>
__global__ void __launch_bounds__(kThreads) prepare_small_kernel(const PrepArgs<NI> args) {
    const PrepParams &p = args.p;
    __shared__ int32_t s_rank[kSmallN], s_start[kSmallN], s_cnt[kSmallN], s_row[kSmallN];
    __shared__ int32_t s_ok[kSmallN], s_comp[kSmallN];
    __shared__ int32_t s_bstart[kSmallN + 1], s_bq[kSmallN];   // by batch position
    __shared__ int32_t s_bad;
    const int tid = threadIdx.x, lane = tid & 31;
    const int n = p.n;
    // as prepare_kernel: the schedule alone is read before the wait when it
    // cannot have been written by the kernel before
    if (!p.early) pdl_wait();
    pdl_trigger();

    if (tid < 32) {
        const bool in = lane < n;
        int32_t c = 0, r = -1;
        if (in) {
            if constexpr (NI > 0) {
                c = args.sched[NI + lane];
                r = args.sched[lane];
            } else {
                c = p.counts[lane];
                r = p.rows[lane];
            }
        }
        const bool bad = __any_sync(0xffffffffu, in && (c < 1 || c > p.T));
        long long tot = in ? c : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        // batch position = requests before this one in (count, schedule
        // index) order; query_start_loc = the sum of their counts
        int32_t rank = 0, start = 0;
        bool repeat = false;
        for (int j = 0; j < n; j++) {
            const int32_t cj = __shfl_sync(0xffffffffu, c, j);
            const int32_t rj = __shfl_sync(0xffffffffu, r, j);
            const bool before = cj < c || (cj == c && j < lane);
            rank += before;
            start += before ? cj : 0;
            repeat |= p.stamp != nullptr && j < lane && rj == r;
        }
        bool ok = in && r >= 0 && r < p.num_rows;
        if (in && !ok) flag(p.err, PKV_DEVERR_ROW);
        if (ok && repeat) {
            ok = false;   // an earlier listing of the row keeps it
            flag(p.err, PKV_DEVERR_DUP);
        }
        if (in && !bad) {
            s_rank[lane] = rank;
            s_start[lane] = start;
            s_cnt[lane] = c;
            s_row[lane] = r;
            s_ok[lane] = ok;
            s_bstart[rank] = start;
            s_bq[rank] = lane;
        }
        if (lane == 0) {
            s_bad = bad || tot != p.T;
            s_bstart[n] = p.T;
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) flag(p.err, PKV_DEVERR_COUNT);
        return;
    }
    if (p.early) pdl_wait();   // from here on the state is read and outputs written

    // per request: completed_tokens, loaded now and used after the full
    // table rows (which do not need it) have gone out
    int32_t comp = 0;
    if (tid < n && s_ok[tid]) comp = p.completed[s_row[tid]];

    // the block-table rows: 16-byte pieces when the rows allow, else entries
    auto table_rows = [&]() {
        for (int g = 0; g < p.G; g++) {
            const int32_t W = p.width[g];
            const bool v4 = W % 4 == 0 &&
                            ((reinterpret_cast<uintptr_t>(p.table[g]) |
                              reinterpret_cast<uintptr_t>(p.out_table[g])) & 15) == 0;
            const int32_t per = v4 ? W / 4 : W;
            for (int32_t f = tid; f < n * per; f += kThreads) {
                const int q = f / per;
                const int32_t e = f - q * per;
                const bool ok = s_ok[q];
                if (p.live_only && ok) {
                    const int64_t len = static_cast<int64_t>(s_comp[q]) + s_cnt[q];
                    const int64_t live = (len + p.bs[g] - 1) / p.bs[g];
                    if (static_cast<int64_t>(e) * (v4 ? 4 : 1) >= live) continue;
                }
                const int64_t src = static_cast<int64_t>(s_row[q]) * W;
                const int64_t dst = static_cast<int64_t>(s_rank[q]) * W;
                if (v4) {
                    const int4 v = ok ? reinterpret_cast<const int4 *>(p.table[g] + src)[e]
                                      : make_int4(-1, -1, -1, -1);
                    reinterpret_cast<int4 *>(p.out_table[g] + dst)[e] = v;
                } else {
                    p.out_table[g][dst + e] = ok ? p.table[g][src + e] : -1;
                }
            }
        }
    };
    if (!p.live_only) table_rows();

    // the batch scalars
    if (tid < n) {
        const bool ok = s_ok[tid];
        const int32_t rank = s_rank[tid];
        s_comp[tid] = comp;
        p.index_mapping[rank] = ok ? s_row[tid] : -1;
        p.qsl[rank] = s_start[tid];
        p.seq_lens[rank] = ok ? comp + s_cnt[tid] : -1;
        if (rank == n - 1) p.qsl[n] = p.T;
    }
    __syncthreads();
    if (p.live_only) table_rows();   // the live entries need completed_tokens

    // per token (batch order)
    for (int32_t t = tid; t < p.T; t += kThreads) {
        int lo = 0, hi = n;   // s_bstart[lo] <= t < s_bstart[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_bstart[mid] <= t) lo = mid; else hi = mid;
        }
        const int q = s_bq[lo];
        const int32_t row = s_row[q];
        const int32_t pos = s_comp[q] + (t - s_bstart[lo]);
        bool ok = s_ok[q];
        if (ok && pos >= p.max_len) {
            flag(p.err, PKV_DEVERR_POSITION);
            ok = false;
        }
        const int32_t id = ok ? ld_stream(p.tokens + row * p.tok_stride + pos) : -1;
        for (int g = 0; g < p.G; g++) {
            int64_t slot = -1;
            if (ok) {
                const int32_t bsz = p.bs[g];
                const int32_t sh = p.bs_shift[g];
                const int32_t lb = sh >= 0 ? (pos >> sh) : pos / bsz;
                const int32_t off = pos - lb * bsz;
                int32_t pb = -1;
                if (lb < p.width[g]) pb = p.table[g][static_cast<int64_t>(row) * p.width[g] + lb];
                if (pb >= 0 && pb < p.num_blocks[g])
                    slot = static_cast<int64_t>(pb) * bsz + off;
                else
                    flag(p.err, PKV_DEVERR_BLOCK);
            }
            p.slots[g][t] = slot;
        }
        p.positions[t] = ok ? pos : -1;
        p.input_ids[t] = id;
    }
}

// ---------------------------------------------------------------------------
// Pure decode steps: T == n, and with every count >= 1 that makes every count
// 1.  Equal counts keep schedule order, so the sort is the identity: request
// i is batch entry i, query_start_loc[i] = i and token i is its one token.
// No staging, scan, slice search or ranks: each CTA takes a contiguous range
// of requests.  After a check that every count is 1 (else nothing is
// written, as in prepare_kernel), the first round of table-row chunks --
// whose sources need only the rows -- goes out with each request's
// completed_tokens load and claim on its row; the stores wait only for the
// claims, and the token id and slot lookups (which need completed_tokens)
// run beside the later rounds.  A row listed twice in a device schedule:
// the first claim to land (an exchange on the row's stamp) keeps it.
// ---------------------------------------------------------------------------
constexpr int kDecodeMaxPer = kThreads;   // requests per CTA, one thread each

template <int CH, int NI>
__global__ void __launch_bounds__(kThreads) prepare_decode_kernel(const PrepArgs<NI> args) {
    const PrepParams &p = args.p;
    constexpr int kRound = 128 / CH > 8 ? 8 : 128 / CH;
    constexpr int kWarpsPerCta = kThreads / 32;
    // s_valid: the row is inside the table (read-only once set); s_ok: and
    // this listing keeps it (set by the request's own thread before the barrier)
    __shared__ int32_t s_row[kDecodeMaxPer], s_valid[kDecodeMaxPer], s_ok[kDecodeMaxPer];
    __shared__ int32_t s_comp[kDecodeMaxPer];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.n, G = p.G;
    const int per = static_cast<int>(p.units_per_cta);   // requests per CTA
    const int i0 = blockIdx.x * per;
    const int nr = min(per, n - i0);
    if (!p.early) pdl_wait();
    pdl_trigger();

    // ---- the schedule: every count 1, this CTA's rows ----------------------
    bool bad = false;
    if constexpr (NI > 0) {
        for (int j = tid; j < n; j += kThreads) bad |= args.sched[NI + j] != 1;
    } else {
        int j = tid;
        if (p.bulk_stage) {   // counts 16-byte aligned
            const int4 *c4 = reinterpret_cast<const int4 *>(p.counts);
            for (; j < n / 4; j += kThreads) {
                const int4 c = ld_stream(c4 + j);
                bad |= (c.x != 1) | (c.y != 1) | (c.z != 1) | (c.w != 1);
            }
            j = (n & ~3) + tid;
        }
        for (; j < n; j += kThreads) bad |= ld_stream(p.counts + j) != 1;
    }
    if (tid < nr) {
        int32_t r;
        if constexpr (NI > 0) r = args.sched[i0 + tid];
        else r = p.rows[i0 + tid];
        s_row[tid] = r;
        s_valid[tid] = r >= 0 && r < p.num_rows;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && tid == 0) flag(p.err, PKV_DEVERR_COUNT);
        return;
    }
    // from here on the state is read and the outputs are written
    if (p.early) pdl_wait();

    // The CTA's full table rows as chunks in (request, group, chunk) order,
    // alpha chunks per request (the host keeps per * alpha below 2^31).  A
    // thread walks chunks tid, tid + kThreads, ... and carries its request q
    // and chunk c within the request along (no division per chunk).
    const int32_t alpha = static_cast<int32_t>(p.alpha);
    const int32_t step_q = kThreads / alpha, step_c = kThreads - step_q * alpha;
    struct Cursor {
        int32_t q, c;
    };
    auto next = [&](Cursor &k) {
        k.q += step_q;
        k.c += step_c;
        if (k.c >= alpha) {
            k.c -= alpha;
            k.q++;
        }
    };
    auto chunk_src = [&](const Cursor &k) -> const char * {
        int g = 0;
        while (k.c >= p.chunk_off[g + 1]) g++;
        return reinterpret_cast<const char *>(p.table[g] +
                                              static_cast<int64_t>(s_row[k.q]) * p.width[g]) +
               static_cast<int64_t>(k.c - p.chunk_off[g]) * CH;
    };
    auto chunk_dst = [&](const Cursor &k) -> char * {
        int g = 0;
        while (k.c >= p.chunk_off[g + 1]) g++;
        return reinterpret_cast<char *>(p.out_table[g] +
                                        static_cast<int64_t>(i0 + k.q) * p.width[g]) +
               static_cast<int64_t>(k.c - p.chunk_off[g]) * CH;
    };
    const Cursor first = {tid / alpha, tid % alpha};
    Chunk<CH> v[kRound];
    Cursor cur = first;
    if (!p.live_only) {   // the first round needs only the rows: in flight now
#pragma unroll
        for (int u = 0; u < kRound; u++) {
            if (cur.q < nr) {
                if (s_valid[cur.q]) ld_chunk(v[u], chunk_src(cur)); else fill_null(v[u]);
            }
            next(cur);
        }
    }

    // ---- per request: completed_tokens and the row's claim -------------------
    int32_t comp = 0;
    bool ok = false;
    int32_t row = -1;
    if (tid < nr) {
        row = s_row[tid];
        ok = s_valid[tid];
        if (ok) {
            comp = p.completed[row];   // used after the barrier (full tables)
            if (p.stamp) {
                // the first exchange on the row's stamp in this call keeps it
                const unsigned long long prev =
                    atomicExch(p.stamp + row, stamp_of(p.gen, i0 + tid));
                if ((prev >> 32) == p.gen) {
                    ok = false;
                    flag(p.err, PKV_DEVERR_DUP);
                }
            }
        } else {
            flag(p.err, PKV_DEVERR_ROW);
        }
        s_ok[tid] = ok;
        if (p.live_only) s_comp[tid] = comp;
    }
    __syncthreads();

    // the request's scalars and its one token
    auto request_outputs = [&]() {
        if (tid >= nr) return;
        const int i = i0 + tid;
        p.index_mapping[i] = ok ? row : -1;
        p.qsl[i] = i;
        if (i == n - 1) p.qsl[n] = n;
        p.seq_lens[i] = ok ? comp + 1 : -1;
        bool tok = ok;
        if (tok && comp >= p.max_len) {
            flag(p.err, PKV_DEVERR_POSITION);
            tok = false;
        }
        p.input_ids[i] = tok ? ld_stream(p.tokens + row * p.tok_stride + comp) : -1;
        for (int g = 0; g < G; g++) {
            int64_t slot = -1;
            if (tok) {
                const int32_t bsz = p.bs[g];
                const int32_t sh = p.bs_shift[g];
                const int32_t lb = sh >= 0 ? (comp >> sh) : comp / bsz;
                const int32_t off = comp - lb * bsz;
                int32_t pb = -1;
                if (lb < p.width[g]) pb = p.table[g][static_cast<int64_t>(row) * p.width[g] + lb];
                if (pb >= 0 && pb < p.num_blocks[g])
                    slot = static_cast<int64_t>(pb) * bsz + off;
                else
                    flag(p.err, PKV_DEVERR_BLOCK);
            }
            p.slots[g][i] = slot;
        }
        p.positions[i] = tok ? comp : -1;
    };

    if (!p.live_only) {
        // ---- block-table rows: the first round's stores, then the rest ---------
        cur = first;
#pragma unroll
        for (int u = 0; u < kRound; u++) {
            if (cur.q < nr) {
                if (!s_ok[cur.q]) fill_null(v[u]);   // loaded before its row was found repeated
                st_chunk(chunk_dst(cur), v[u]);
            }
            next(cur);
        }
        request_outputs();
        while (cur.q < nr) {
            const Cursor round = cur;
#pragma unroll
            for (int u = 0; u < kRound; u++) {
                if (cur.q < nr) {
                    if (s_ok[cur.q]) ld_chunk(v[u], chunk_src(cur)); else fill_null(v[u]);
                }
                next(cur);
            }
            cur = round;
#pragma unroll
            for (int u = 0; u < kRound; u++) {
                if (cur.q < nr) st_chunk(chunk_dst(cur), v[u]);
                next(cur);
            }
        }
    } else {
        request_outputs();
        // the live entries, j < ceil((completed + 1) / bs), a warp per request
        for (int q = warp; q < nr; q += kWarpsPerCta) {
            const bool q_ok = s_ok[q];
            const int64_t len = static_cast<int64_t>(s_comp[q]) + 1;
            for (int g = 0; g < G; g++) {
                const int64_t nb = (len + p.bs[g] - 1) / p.bs[g];
                const int64_t live = nb < p.width[g] ? nb : p.width[g];
                const int32_t nch = static_cast<int32_t>((live * 4 + CH - 1) / CH);
                const char *src = reinterpret_cast<const char *>(
                    p.table[g] + static_cast<int64_t>(s_row[q]) * p.width[g]);
                char *dst = reinterpret_cast<char *>(p.out_table[g] +
                                                     static_cast<int64_t>(i0 + q) * p.width[g]);
                for (int32_t k0 = 0; k0 < nch; k0 += 32 * kRound) {
#pragma unroll
                    for (int u = 0; u < kRound; u++) {
                        const int32_t k = k0 + u * 32 + lane;
                        if (k < nch) {
                            if (q_ok) ld_chunk(v[u], src + static_cast<int64_t>(k) * CH);
                            else fill_null(v[u]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kRound; u++) {
                        const int32_t k = k0 + u * 32 + lane;
                        if (k < nch) st_chunk(dst + static_cast<int64_t>(k) * CH, v[u]);
                    }
                }
            }
        }
    }
}

__global__ void advance_kernel(const int32_t *rows, const int32_t *counts, int32_t n,
                               int32_t num_rows, int32_t *completed) {
    pdl_wait();   // the batch build reads completed_tokens first
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const int32_t r = rows[i];
        if (r >= 0 && r < num_rows) completed[r] += counts[i];
    }
}

size_t prepare_smem_bytes(int32_t n) {
    return static_cast<size_t>(smem_layout(n).words) * sizeof(int32_t);
}

int ensure_kernel_attributes(int device) {
    static int configured[64] = {0};
    if (device < 0 || device >= 64) return PKV_ERR_INVALID_ARG;
    if (!configured[device]) {
        const int bytes = static_cast<int>(prepare_smem_bytes(PKV_MAX_BATCH));
        const void *kernels[] = {
            reinterpret_cast<const void *>(prepare_kernel<4, 0>),
            reinterpret_cast<const void *>(prepare_kernel<16, 0>),
            reinterpret_cast<const void *>(prepare_kernel<32, 0>),
            reinterpret_cast<const void *>(prepare_kernel<4, kInlineSmall>),
            reinterpret_cast<const void *>(prepare_kernel<16, kInlineSmall>),
            reinterpret_cast<const void *>(prepare_kernel<32, kInlineSmall>),
            reinterpret_cast<const void *>(prepare_kernel<4, kInlineMax>),
            reinterpret_cast<const void *>(prepare_kernel<16, kInlineMax>),
            reinterpret_cast<const void *>(prepare_kernel<32, kInlineMax>)};
        for (const void *k : kernels)
            PKV_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
        configured[device] = 1;
    }
    return PKV_OK;
}

bool aligned_to(const void *q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; }

// Resident CTAs per SM of prepare_kernel<CH, NI> with `smem` bytes of dynamic
// shared memory, from the occupancy calculator, cached per device in 1 KB
// steps of shared memory (each step computed for its upper end, so a cached
// figure never exceeds the true one).  The library is single-threaded per
// its contract, so the cache needs no lock.
template <int CH, int NI>
cudaError_t resident_ctas(int device, size_t smem, int *out) {
    static std::unordered_map<uint64_t, int> cache;
    const size_t cap = prepare_smem_bytes(PKV_MAX_BATCH);
    const uint64_t step = (smem + 1023) / 1024;
    const uint64_t key = (static_cast<uint64_t>(device) << 32) | step;
    const auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    size_t upper = static_cast<size_t>(step) * 1024;
    if (upper > cap) upper = cap;
    if (upper < smem) upper = smem;
    int b = 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, prepare_kernel<CH, NI>, kThreads, upper);
    if (e != cudaSuccess) return e;
    if (b < 1) b = 1;
    cache.emplace(key, b);
    *out = b;
    return cudaSuccess;
}

// Given PrepParams with pointers, sizes and per-group widths, block sizes,
// pools and tables filled in: choose the chunk width (32 bytes when every
// source and destination table row starts 32-byte aligned, else 16, else 4),
// lay out the unit space, size the grid to the SMs, and launch.
template <int CH, int NI>
int launch_with(PrepParams &p, const int32_t *h_rows, const int32_t *h_counts, int device,
                int num_sms, cudaStream_t s) {
    const size_t smem = prepare_smem_bytes(p.n);
    int per_sm = 0;
    PKV_CUDA_TRY((resident_ctas<CH, NI>(device, smem, &per_sm)));
    const int64_t max_ctas = static_cast<int64_t>(num_sms) * per_sm;
    int64_t per_cta = (p.total_units + max_ctas - 1) / max_ctas;
    if (per_cta < kMinUnitsPerCta) per_cta = kMinUnitsPerCta;
    p.units_per_cta = per_cta;
    const int64_t grid = (p.total_units + per_cta - 1) / per_cta;
    PrepArgs<NI> a;
    a.p = p;
    if constexpr (NI > 0) {
        memcpy(a.sched, h_rows, static_cast<size_t>(p.n) * sizeof(int32_t));
        memcpy(a.sched + NI, h_counts, static_cast<size_t>(p.n) * sizeof(int32_t));
    }
    PKV_CUDA_TRY(launch_pdl(prepare_kernel<CH, NI>, dim3(static_cast<unsigned>(grid)),
                            dim3(kThreads), smem, s, a));
    return PKV_OK;
}

// Resident CTAs per SM of prepare_decode_kernel<CH, NI> (static shared
// memory only), from the occupancy calculator, cached per device.
template <int CH, int NI>
cudaError_t decode_resident_ctas(int device, int *out) {
    static int cache[64] = {0};
    if (device >= 0 && device < 64 && cache[device]) {
        *out = cache[device];
        return cudaSuccess;
    }
    int b = 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, prepare_decode_kernel<CH, NI>, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (b < 1) b = 1;
    if (device >= 0 && device < 64) cache[device] = b;
    *out = b;
    return cudaSuccess;
}

// A pure decode step (T == n): contiguous ranges of requests per CTA, at
// least one table-row chunk per thread, at most one wave of CTAs.
template <int CH, int NI>
int launch_decode_with(PrepParams &p, const int32_t *h_rows, const int32_t *h_counts, int device,
                       int num_sms, cudaStream_t s) {
    int per_sm = 0;
    PKV_CUDA_TRY((decode_resident_ctas<CH, NI>(device, &per_sm)));
    const int64_t max_ctas = static_cast<int64_t>(num_sms) * per_sm;
    int64_t per = (kThreads + p.alpha - 1) / p.alpha;
    const int64_t spread = (p.n + max_ctas - 1) / max_ctas;
    if (per < spread) per = spread;
    if (per > kDecodeMaxPer) per = kDecodeMaxPer;
    if (per * p.alpha > INT32_MAX) per = INT32_MAX / p.alpha;   // 32-bit chunk indexes
    if (per < 1) return PKV_ERR_INVALID_ARG;
    p.units_per_cta = per;
    const int64_t grid = (p.n + per - 1) / per;
    PrepArgs<NI> a;
    a.p = p;
    if constexpr (NI > 0) {
        memcpy(a.sched, h_rows, static_cast<size_t>(p.n) * sizeof(int32_t));
        memcpy(a.sched + NI, h_counts, static_cast<size_t>(p.n) * sizeof(int32_t));
    }
    PKV_CUDA_TRY(launch_pdl(prepare_decode_kernel<CH, NI>, dim3(static_cast<unsigned>(grid)),
                            dim3(kThreads), 0, s, a));
    return PKV_OK;
}

template <int CH>
int launch_chunked(PrepParams &p, const int32_t *h_rows, const int32_t *h_counts, int device,
                   int num_sms, cudaStream_t s) {
    int64_t alpha = 0;
    p.chunk_off[0] = 0;
    for (int g = 0; g < p.G; g++) {
        const int32_t units = static_cast<int32_t>(static_cast<int64_t>(p.width[g]) * 4 / CH);
        p.chunk_off[g + 1] = p.chunk_off[g] + units;
        alpha += units;
    }
    for (int g = p.G; g < PKV_MAX_GROUPS; g++) p.chunk_off[g + 1] = p.chunk_off[g];
    p.alpha = alpha;
    p.total_units = alpha * p.n + p.T;
    if (p.T == p.n) {   // every count 1 (or the kernel finds a count error)
        if (!h_rows) return launch_decode_with<CH, 0>(p, nullptr, nullptr, device, num_sms, s);
        if (p.n <= kInlineSmall)
            return launch_decode_with<CH, kInlineSmall>(p, h_rows, h_counts, device, num_sms, s);
        return launch_decode_with<CH, kInlineMax>(p, h_rows, h_counts, device, num_sms, s);
    }
    if (!h_rows) return launch_with<CH, 0>(p, nullptr, nullptr, device, num_sms, s);
    if (p.n <= kInlineSmall)
        return launch_with<CH, kInlineSmall>(p, h_rows, h_counts, device, num_sms, s);
    return launch_with<CH, kInlineMax>(p, h_rows, h_counts, device, num_sms, s);
}

// h_rows / h_counts: a host schedule of at most kInlineMax requests to pass in
// the kernel's parameters, or null (the schedule is at p.rows / p.counts).
int launch_params(PrepParams &p, const int32_t *h_rows, const int32_t *h_counts, int device,
                  int num_sms, cudaStream_t s) {
    int rc = ensure_kernel_attributes(device);
    if (rc != PKV_OK) return rc;
    if (h_rows && (p.n > kInlineMax || !h_counts)) return PKV_ERR_INVALID_ARG;
    p.bulk_stage = !h_rows && aligned_to(p.counts, 16) && aligned_to(p.rows, 16);
    int ch = 32;
    for (int g = 0; g < p.G; g++) {
        const int64_t row_bytes = static_cast<int64_t>(p.width[g]) * 4;
        if (row_bytes % 32 || !aligned_to(p.table[g], 32) || !aligned_to(p.out_table[g], 32))
            ch = ch > 16 ? 16 : ch;
        if (row_bytes % 16 || !aligned_to(p.table[g], 16) || !aligned_to(p.out_table[g], 16))
            ch = 4;
    }
    for (int g = 0; g < p.G; g++) {
        int sh = -1;
        if ((p.bs[g] & (p.bs[g] - 1)) == 0) {
            sh = 0;
            while ((1 << sh) < p.bs[g]) sh++;
        }
        p.bs_shift[g] = sh;
    }
    int64_t entries = 0;
    for (int g = 0; g < p.G; g++) entries += p.width[g];
    if (p.n <= kSmallN && p.T <= kSmallT && p.n * entries <= kSmallEntries) {
        if (h_rows) {
            PrepArgs<kInlineSmall> a;
            a.p = p;
            memcpy(a.sched, h_rows, static_cast<size_t>(p.n) * sizeof(int32_t));
            memcpy(a.sched + kInlineSmall, h_counts, static_cast<size_t>(p.n) * sizeof(int32_t));
            PKV_CUDA_TRY(launch_pdl(prepare_small_kernel<kInlineSmall>, dim3(1), dim3(kThreads), 0, s, a));
        } else {
            PrepArgs<0> a;
            a.p = p;
            PKV_CUDA_TRY(launch_pdl(prepare_small_kernel<0>, dim3(1), dim3(kThreads), 0, s, a));
        }
        return PKV_OK;
    }
    if (ch == 32) return launch_chunked<32>(p, h_rows, h_counts, device, num_sms, s);
    if (ch == 16) return launch_chunked<16>(p, h_rows, h_counts, device, num_sms, s);
    return launch_chunked<4>(p, h_rows, h_counts, device, num_sms, s);
}

// Parameters of one batch build from a request-state table; with h_rows /
// h_counts (at most kInlineMax requests) the schedule travels in the kernel's
// parameters and in.d_rows / in.d_counts are not read.
int launch_prepare_from(pkv_state *st, const pkv::PrepareLaunch &in, const int32_t *h_rows,
                        const int32_t *h_counts, const pkv_batch_out *out, cudaStream_t s) {
    PrepParams p = {};
    p.rows = in.d_rows;
    p.counts = in.d_counts;
    p.n = in.n;
    p.T = in.total_tokens;
    p.live_only = (in.flags & PKV_LIVE_TABLES) != 0;
    p.early = h_rows != nullptr || !in.device_schedule || (in.flags & PKV_SCHEDULE_SETTLED) != 0;
    p.num_rows = st->rows;
    p.max_len = st->max_len;
    p.G = st->num_groups;
    p.tok_stride = st->max_len;
    p.completed = st->d_completed;
    p.tokens = st->d_tokens;
    p.index_mapping = out->index_mapping;
    p.qsl = out->query_start_loc;
    p.seq_lens = out->seq_lens;
    p.positions = out->positions;
    p.input_ids = out->input_ids;
    p.err = st->d_error;
    if (in.device_schedule) {
        if (++st->stamp_gen == 0) {
            PKV_CUDA_TRY(cudaMemsetAsync(st->d_stamp, 0,
                                         static_cast<size_t>(st->rows) * sizeof(unsigned long long), s));
            st->stamp_gen = 1;
        }
        p.stamp = st->d_stamp;
        p.gen = st->stamp_gen;
    }
    for (int g = 0; g < st->num_groups; g++) {
        const pkv::GroupState &gs = st->groups[g];
        p.width[g] = gs.width;
        p.bs[g] = gs.block_size;
        p.num_blocks[g] = gs.num_blocks;
        p.table[g] = gs.d_table;
        p.out_table[g] = out->block_tables[g];
        p.slots[g] = out->slot_mapping[g];
    }
    return launch_params(p, h_rows, h_counts, st->device, st->num_sms, s);
}

// Device staging of host schedules too large for the launch parameters:
// two buffers used in turn, filled by a copy stream of the state's own.  The
// copy of a call starts as soon as the call is made -- overlapping the GPU
// work already queued on the caller's stream -- and waits only for the
// kernels of the call before the last one (the last readers of its buffer);
// the caller's stream waits for the copy before the prepare kernel.
struct StageSide {
    cudaStream_t copy = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
    int32_t *d_buf[2] = {nullptr, nullptr};
    int slot = 0;
};
std::unordered_map<const pkv_state *, StageSide> g_stage;   // single-threaded library

void free_stage(StageSide &sd) {
    if (sd.copy) cudaStreamSynchronize(sd.copy);
    for (int k = 0; k < 2; k++) {
        if (sd.copied[k]) cudaEventDestroy(sd.copied[k]);
        if (sd.consumed[k]) cudaEventDestroy(sd.consumed[k]);
        if (sd.d_buf[k]) cudaFree(sd.d_buf[k]);
    }
    if (sd.copy) cudaStreamDestroy(sd.copy);
    sd = StageSide();
}

int stage_side(const pkv_state *st, StageSide **out) {
    auto it = g_stage.find(st);
    if (it != g_stage.end()) {
        *out = &it->second;
        return PKV_OK;
    }
    StageSide sd;
    const size_t bytes = static_cast<size_t>(2 * (PKV_MAX_BATCH + 4)) * sizeof(int32_t);
    cudaError_t e = cudaStreamCreateWithFlags(&sd.copy, cudaStreamNonBlocking);
    for (int k = 0; k < 2 && e == cudaSuccess; k++) {
        e = cudaEventCreateWithFlags(&sd.copied[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.consumed[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaMalloc(&sd.d_buf[k], bytes);
    }
    if (e != cudaSuccess) {
        free_stage(sd);
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    *out = &g_stage.emplace(st, sd).first->second;
    return PKV_OK;
}

}  // namespace

namespace pkv {

// Called by pkv_state_destroy: the state's staging stream, events and buffers.
void release_prepare_staging(const pkv_state *st) {
    auto it = g_stage.find(st);
    if (it == g_stage.end()) return;
    free_stage(it->second);
    g_stage.erase(it);
}

int launch_prepare(pkv_state *st, const PrepareLaunch &in, const pkv_batch_out *out,
                   cudaStream_t s) {
    return launch_prepare_from(st, in, nullptr, nullptr, out, s);
}

int launch_advance(pkv_state *st, const int32_t *d_rows, const int32_t *d_counts, int32_t n,
                   cudaStream_t s) {
    PKV_CUDA_TRY(launch_pdl(advance_kernel, dim3((n + 255) / 256), dim3(256), 0, s, d_rows, d_counts,
                            n, st->rows, st->d_completed));
    return PKV_OK;
}

}  // namespace pkv

static bool outputs_ok(const pkv_state *st, const pkv_batch_out *out, int32_t n, int64_t T) {
    if (!out) return false;
    if (n > 0 && (!out->index_mapping || !out->seq_lens)) return false;
    if (!out->query_start_loc) return false;
    if (T > 0 && (!out->positions || !out->input_ids)) return false;
    for (int g = 0; g < st->num_groups; g++) {
        if (n > 0 && !out->block_tables[g]) return false;
        if (T > 0 && !out->slot_mapping[g]) return false;
    }
    return true;
}

extern "C" {

int pkv_prepare_batch(pkv_state *st, const int32_t *rows, const int32_t *num_sched, int32_t n,
                      int32_t flags, const pkv_batch_out *out, int32_t *out_total_tokens,
                      pkv_stream_t stream) {
    if (!st || !out_total_tokens) return PKV_ERR_INVALID_ARG;
    if (n < 0 || n > PKV_MAX_BATCH || n > st->rows) return PKV_ERR_INVALID_ARG;
    if (flags & ~(PKV_ADVANCE | PKV_LIVE_TABLES)) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!rows || !num_sched)) return PKV_ERR_INVALID_ARG;
    // validate the schedule against the host mirrors
    if (++st->seen_gen == 0) {
        std::fill(st->seen.begin(), st->seen.end(), 0u);
        st->seen_gen = 1;
    }
    int64_t T = 0;
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        if (st->seen[r] == st->seen_gen) return PKV_ERR_INVALID_ARG;
        st->seen[r] = st->seen_gen;
        const int32_t c = num_sched[i];
        if (c < 1) return PKV_ERR_INVALID_ARG;
        const int64_t end = static_cast<int64_t>(st->completed[r]) + c;
        if (end > st->ntok[r]) return PKV_ERR_CAPACITY;
        for (int g = 0; g < st->num_groups; g++) {
            const pkv::GroupState &gs = st->groups[g];
            const int64_t first = st->completed[r] / gs.block_size;
            const int64_t last = (end - 1) / gs.block_size;
            if (last >= gs.nblk[r] || first < gs.lead_null[r]) return PKV_ERR_CAPACITY;
        }
        T += c;
    }
    if (T >= PKV_MAX_TOKENS) return PKV_ERR_INVALID_ARG;
    if (!outputs_ok(st, out, n, T)) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = pkv::as_stream(stream);
    if (n == 0) {
        PKV_CUDA_TRY(cudaMemsetAsync(out->query_start_loc, 0, sizeof(int32_t), s));
        *out_total_tokens = 0;
        return PKV_OK;
    }
    if (n <= kInlineMax && !(flags & PKV_ADVANCE)) {
        // the schedule travels in the kernel's parameters: no staging copy
        const pkv::PrepareLaunch in{nullptr, nullptr, n, static_cast<int32_t>(T), flags};
        const int rc = launch_prepare_from(st, in, rows, num_sched, out, s);
        if (rc != PKV_OK) return rc;
        *out_total_tokens = static_cast<int32_t>(T);
        return PKV_OK;
    }
    // one host-to-device copy: rows, then counts at a 16-byte aligned offset
    const int32_t n4 = (n + 3) & ~3;
    const size_t bytes = static_cast<size_t>(n4 + n) * 4;
    int status;
    char *buf = st->ring.reserve(bytes, &status);
    if (!buf) return status;
    memcpy(buf, rows, static_cast<size_t>(n) * 4);
    memcpy(buf + static_cast<size_t>(n4) * 4, num_sched, static_cast<size_t>(n) * 4);
    // off the caller's stream unless it is being captured into a graph (a
    // captured stream may not wait on work outside the capture)
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusActive;   // unknown: stay on the caller's stream
    }
    StageSide *sd = nullptr;
    if (cap == cudaStreamCaptureStatusNone) {
        const int rc0 = stage_side(st, &sd);
        if (rc0 != PKV_OK) return rc0;
    }
    int32_t *dst = st->d_sched;
    cudaStream_t cs = s;
    int slot = 0;
    if (sd) {
        slot = sd->slot;
        sd->slot ^= 1;
        dst = sd->d_buf[slot];
        cs = sd->copy;
        PKV_CUDA_TRY(cudaStreamWaitEvent(cs, sd->consumed[slot], 0));
    }
    cudaError_t e = cudaMemcpyAsync(dst, buf, bytes, cudaMemcpyHostToDevice, cs);
    int rc = st->ring.fence(cs);
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    if (sd) {
        PKV_CUDA_TRY(cudaEventRecord(sd->copied[slot], cs));
        PKV_CUDA_TRY(cudaStreamWaitEvent(s, sd->copied[slot], 0));
    }
    pkv::PrepareLaunch in{dst, dst + n4, n, static_cast<int32_t>(T), flags};
    rc = pkv::launch_prepare(st, in, out, s);
    if (rc != PKV_OK) return rc;
    if (flags & PKV_ADVANCE) {
        rc = pkv::launch_advance(st, in.d_rows, in.d_counts, n, s);
        if (rc != PKV_OK) return rc;
        for (int32_t i = 0; i < n; i++) st->completed[rows[i]] += num_sched[i];
    }
    // the staged buffer is free again once these kernels have run
    if (sd) PKV_CUDA_TRY(cudaEventRecord(sd->consumed[slot], s));
    *out_total_tokens = static_cast<int32_t>(T);
    return PKV_OK;
}

int pkv_prepare_batch_device(pkv_state *st, const int32_t *d_rows, const int32_t *d_num_sched,
                             int32_t n, int32_t total_tokens, int32_t flags,
                             const pkv_batch_out *out, pkv_stream_t stream) {
    if (!st) return PKV_ERR_INVALID_ARG;
    if (flags & ~(PKV_LIVE_TABLES | PKV_SCHEDULE_SETTLED)) return PKV_ERR_INVALID_ARG;
    if (n < 0 || n > PKV_MAX_BATCH || total_tokens < 0 || total_tokens >= PKV_MAX_TOKENS)
        return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!d_rows || !d_num_sched)) return PKV_ERR_INVALID_ARG;
    if (!outputs_ok(st, out, n, total_tokens)) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = pkv::as_stream(stream);
    if (n == 0) {
        PKV_CUDA_TRY(cudaMemsetAsync(out->query_start_loc, 0, sizeof(int32_t), s));
        return PKV_OK;
    }
    pkv::PrepareLaunch in{d_rows, d_num_sched, n, total_tokens, flags, 1};
    return pkv::launch_prepare(st, in, out, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Batch build that allocates nothing: pkv_prepare_batch_static.
//
// The regular host-schedule entry point stages the schedule in memory that
// pkv_state_create allocated.  This variant takes the request-state table as
// caller-owned device arrays and allocates nothing: a schedule of up to
// kInlineMax requests travels in the kernel's parameter block, and a larger
// one is staged in a fixed device array compiled into the library.  That
// array is shared by every call on a device and keeps the last call's
// contents; nothing in it has to start at zero, because each call overwrites
// the [0, n) entries the kernel reads before launching.
// ---------------------------------------------------------------------------
namespace {

// rows at [0, n), counts at the 16-byte aligned offset round_up(n, 4)
static __device__ __align__(256) int32_t g_static_schedule[2 * (PKV_STATIC_MAX_BATCH + 4)];

// The same layout in ordinary (pageable) host memory.  A host-to-device
// cudaMemcpyAsync from pageable memory returns only once the bytes have been
// taken in by the driver, so the caller's arrays -- pinned or not -- and this
// buffer may be reused as soon as the call returns.
int32_t g_static_host[2 * (PKV_STATIC_MAX_BATCH + 4)];

// Repeated-row check without allocating: open addressing over twice the
// largest batch, entries valid only when stamped with the current call.
constexpr uint32_t kDupSlots = 2 * PKV_STATIC_MAX_BATCH;   // a power of two
static_assert((kDupSlots & (kDupSlots - 1)) == 0, "kDupSlots must be a power of two");
int32_t g_dup_row[kDupSlots];
uint32_t g_dup_stamp[kDupSlots];
uint32_t g_dup_gen = 0;

bool has_repeated_row(const int32_t *rows, int32_t n) {
    if (++g_dup_gen == 0) {
        memset(g_dup_stamp, 0, sizeof(g_dup_stamp));
        g_dup_gen = 1;
    }
    for (int32_t i = 0; i < n; i++) {
        uint32_t h = (static_cast<uint32_t>(rows[i]) * 2654435761u) & (kDupSlots - 1);
        while (g_dup_stamp[h] == g_dup_gen) {
            if (g_dup_row[h] == rows[i]) return true;
            h = (h + 1) & (kDupSlots - 1);
        }
        g_dup_stamp[h] = g_dup_gen;
        g_dup_row[h] = rows[i];
    }
    return false;
}

}  // namespace

extern "C" int pkv_prepare_batch_static(
    const int32_t *d_completed, const int32_t *d_token_ids, int32_t max_reqs,
    int32_t max_model_len, int32_t num_groups, const pkv_group_spec *groups,
    const int32_t *const *d_block_tables, const int32_t *rows, const int32_t *num_sched,
    int32_t n, const pkv_batch_out *out, int32_t *d_error, int32_t *out_total_tokens,
    pkv_stream_t stream) {
    if (!d_completed || !d_token_ids || !groups || !d_block_tables || !out || !out_total_tokens)
        return PKV_ERR_INVALID_ARG;
    if (max_reqs < 1 || max_model_len < 1 || num_groups < 1 || num_groups > PKV_MAX_GROUPS)
        return PKV_ERR_INVALID_ARG;
    if (n < 0 || n > PKV_STATIC_MAX_BATCH || n > max_reqs) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!rows || !num_sched)) return PKV_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; g++) {
        if (groups[g].block_size < 1 || groups[g].max_blocks_per_req < 1 ||
            groups[g].num_blocks < 1 || groups[g].num_blocks > INT32_MAX || !d_block_tables[g])
            return PKV_ERR_INVALID_ARG;
    }
    int64_t T = 0;
    for (int32_t i = 0; i < n; i++) {
        if (rows[i] < 0 || rows[i] >= max_reqs || num_sched[i] < 1) return PKV_ERR_INVALID_ARG;
        T += num_sched[i];
    }
    if (T >= PKV_MAX_TOKENS) return PKV_ERR_INVALID_ARG;
    // one batch row per request: a row listed twice would give two requests
    // the same slots
    if (has_repeated_row(rows, n)) return PKV_ERR_INVALID_ARG;
    if (!out->query_start_loc || (n > 0 && (!out->index_mapping || !out->seq_lens)) ||
        (T > 0 && (!out->positions || !out->input_ids)))
        return PKV_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; g++) {
        if ((n > 0 && !out->block_tables[g]) || (T > 0 && !out->slot_mapping[g]))
            return PKV_ERR_INVALID_ARG;
    }
    cudaStream_t s = pkv::as_stream(stream);
    if (n == 0) {
        PKV_CUDA_TRY(cudaMemsetAsync(out->query_start_loc, 0, sizeof(int32_t), s));
        *out_total_tokens = 0;
        return PKV_OK;
    }
    int device = 0;
    PKV_CUDA_TRY(cudaGetDevice(&device));
    int num_sms = 0;
    PKV_CUDA_TRY(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device));

    PrepParams p = {};
    p.n = n;
    p.T = static_cast<int32_t>(T);
    p.num_rows = max_reqs;
    p.max_len = max_model_len;
    p.G = num_groups;
    p.tok_stride = max_model_len;
    p.completed = d_completed;
    p.tokens = d_token_ids;
    p.index_mapping = out->index_mapping;
    p.qsl = out->query_start_loc;
    p.seq_lens = out->seq_lens;
    p.positions = out->positions;
    p.input_ids = out->input_ids;
    p.err = d_error;
    p.early = 1;   // the schedule comes in the parameters or by a copy on s
    for (int g = 0; g < num_groups; g++) {
        p.width[g] = groups[g].max_blocks_per_req;
        p.bs[g] = groups[g].block_size;
        p.num_blocks[g] = groups[g].num_blocks;
        p.table[g] = d_block_tables[g];
        p.out_table[g] = out->block_tables[g];
        p.slots[g] = out->slot_mapping[g];
    }
    int rc;
    if (n <= kInlineMax) {
        // in the kernel's parameters: no copy, the fixed array is not used
        rc = launch_params(p, rows, num_sched, device, num_sms, s);
    } else {
        // a copy recorded into a graph would read the host buffer again at
        // every replay, after later calls have overwritten it
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        PKV_CUDA_TRY(cudaStreamIsCapturing(s, &cap));
        if (cap != cudaStreamCaptureStatusNone) return PKV_ERR_INVALID_ARG;
        // In host code g_static_schedule only stands in for the array; its
        // device address (looked up on every call, so that it is never stale)
        // is what the copy and the kernel use.
        void *sym = nullptr;
        PKV_CUDA_TRY(cudaGetSymbolAddress(&sym, g_static_schedule));
        int32_t *sched = static_cast<int32_t *>(sym);
        const int32_t n4 = (n + 3) & ~3;
        memcpy(g_static_host, rows, static_cast<size_t>(n) * 4);
        memset(g_static_host + n, 0, static_cast<size_t>(n4 - n) * 4);
        memcpy(g_static_host + n4, num_sched, static_cast<size_t>(n) * 4);
        PKV_CUDA_TRY(cudaMemcpyAsync(sched, g_static_host, static_cast<size_t>(n4 + n) * 4,
                                     cudaMemcpyHostToDevice, s));
        p.rows = sched;
        p.counts = sched + n4;
        rc = launch_params(p, nullptr, nullptr, device, num_sms, s);
    }
    if (rc != PKV_OK) return rc;
    *out_total_tokens = static_cast<int32_t>(T);
    return PKV_OK;
}

// ---------------------------------------------------------------------------
// pkv_selftest_wait_timeout: a wait that nothing completes, ended by its own
// poll limit (the give-up path of the kernels' bounded waits).
// ---------------------------------------------------------------------------
namespace {

__global__ void wait_timeout_kernel(int32_t *err, uint32_t polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // one arrival expected; none comes
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, polls)) flag(err, PKV_DEVERR_TIMEOUT);
}

}  // namespace

int pkv_selftest_wait_timeout(int32_t *d_error, uint32_t polls, pkv_stream_t stream) {
    if (!d_error || polls < 1 || polls > 1000000) return PKV_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, pkv::as_stream(stream)>>>(d_error, polls);
    PKV_CUDA_TRY(cudaGetLastError());
    return PKV_OK;
}
