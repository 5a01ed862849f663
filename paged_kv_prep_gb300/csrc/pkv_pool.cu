// Free-block pools and allocate_slots.
//
// "allocate_slots()" section of "从源码读 vLLM Scheduler": for one request,
// in order -- count the slots needed (computed + new + speculative lookahead),
// free the sliding-window blocks no longer needed, count the new blocks
// actually missing, keep a watermark in reserve and refuse if
// required = new + watermark exceeds available = free - reserved, otherwise
// allocate.  The scheduler stops at a refused request.
//
// Readings (the same as the CPU oracle's): one call is a batch of requests,
// each taken through all five steps before the next; the first refused
// request and all after it are not admitted, and the refused request's window
// frees stand (they precede its check); "reserved" is 0; each group's free
// ids form a stack: frees are pushed lowest logical block first, allocations
// pop from the top (so a request's own frees, and earlier requests', can
// serve it); blocks wholly before max(0, computed - (window - 1)) are out of
// the window.
//
// GB300 design: the sequential stack is never simulated.  A one-CTA plan
// kernel computes every request's frees f and missing blocks a per group,
// scans f - a into S_i (the stack height before request i), finds the first
// request whose a + watermark exceeds S_i + f_i, and the suffix minima of S.
// Then, without any ordering between requests: the id request i pops at
// stack position p is its own freed id when p >= S_i, else the id pushed
// there by the latest earlier request m with S_m <= p (that request must
// have pushed p, and the stack stayed above p since), else the id the stack
// held at the start (pop kernel, one warp per request and group, walking
// back over S with a running minimum).  A pushed id survives in the final
// stack when no later processed request starts at or below its position
// (push kernel).  The host only validates the call, stages it and, after the
// kernels, copies the per-request results into its mirrors.
#include <string.h>

#include <algorithm>
#include <vector>

#include "pkv_async.cuh"
#include "pkv_common.cuh"

namespace {

using namespace pkv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// dst[k] = src[k * step] for k < count; then src[k * step] = -1 if clear.
struct MoveOp {
    int32_t *dst;
    int32_t *src;
    int32_t count;
    int32_t step;
    int32_t clear;
    int32_t pad;
};
static_assert(sizeof(MoveOp) == 32, "MoveOp layout");

__global__ void __launch_bounds__(kThreads) move_kernel(const MoveOp *ops, int32_t nops) {
    pdl_wait();   // pops must read the stack before the pushes overwrite it
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); w < nops;
         w += stride) {
        const MoveOp op = ops[w];
        for (int32_t k = lane; k < op.count; k += 32) {
            int32_t *s = op.src + static_cast<int64_t>(k) * op.step;
            op.dst[k] = *s;
            if (op.clear) *s = -1;
        }
    }
}

// Stage `ops` through the pinned ring into st->d_apply and launch one move.
int launch_moves(pkv_state *st, const std::vector<MoveOp> &ops, cudaStream_t s) {
    const size_t per = stage_limit(st) / sizeof(MoveOp);
    for (size_t a = 0; a < ops.size(); a += per) {
        const size_t m = std::min(per, ops.size() - a);
        int status;
        char *buf = st->ring.reserve(m * sizeof(MoveOp), &status);
        if (!buf) return status;
        memcpy(buf, ops.data() + a, m * sizeof(MoveOp));
        cudaError_t e = cudaMemcpyAsync(st->d_apply, buf, m * sizeof(MoveOp),
                                        cudaMemcpyHostToDevice, s);
        const int rc = st->ring.fence(s);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return PKV_ERR_CUDA;
        }
        if (rc != PKV_OK) return rc;
        const int64_t need = (static_cast<int64_t>(m) + kWarps - 1) / kWarps;
        const int64_t wave = static_cast<int64_t>(st->num_sms) * (2048 / kThreads);
        const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
        PKV_CUDA_TRY(launch_pdl(move_kernel, dim3(grid), dim3(kThreads), 0, s,
                                reinterpret_cast<const MoveOp *>(st->d_apply),
                                static_cast<int32_t>(m)));
    }
    return PKV_OK;
}

// ---- device allocate_slots --------------------------------------------------

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kResWords = 16;   // status, admitted, processed, pad..., top[g] at 8 + g

enum : int32_t { kAllocOk = 0, kAllocTooLong = 1, kAllocStackFull = 2 };

struct AllocParams {
    const int32_t *rows, *num_new, *lookahead;   // [n]
    const int32_t *have, *lead;                  // [G][n]: blocks held, leading -1 entries
    const int32_t *completed;                    // state's completed_tokens
    int32_t *S, *suf, *F, *A;                    // [G][n]
    int32_t *res;                                // [kResWords]
    int32_t n, G, watermark, pad;
    int32_t bs[PKV_MAX_GROUPS], W[PKV_MAX_GROUPS], window[PKV_MAX_GROUPS];
    int32_t c0[PKV_MAX_GROUPS], cap[PKV_MAX_GROUPS];
    int32_t *table[PKV_MAX_GROUPS];
    int32_t *pool[PKV_MAX_GROUPS];
};

// Exclusive prefix sum over the CTA in thread order.
__device__ __forceinline__ long long cta_excl_sum(long long v, long long *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = sm[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sm[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const long long before = warp ? sm[warp - 1] : 0;
    const long long out = before + x - v;
    __syncthreads();   // sm is reused by the next call
    return out;
}

// Minimum over the threads after this one (thread order), `init` if none.
__device__ __forceinline__ int32_t cta_suffix_min_excl(int32_t v, int32_t init, int32_t *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x = min(x, y);
    }
    // x = min over lanes >= lane of this warp
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = sm[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_down_sync(0xffffffffu, w, o);
            if (lane + o < 32) w = min(w, y);
        }
        sm[lane] = w;   // min over warps >= lane
    }
    __syncthreads();
    int32_t after = __shfl_down_sync(0xffffffffu, x, 1);
    if (lane == 31) after = INT32_MAX;
    const int32_t later_warps = warp + 1 < kPlanWarps ? sm[warp + 1] : INT32_MAX;
    const int32_t out = min(init, min(after, later_warps));
    __syncthreads();
    return out;
}

__device__ __forceinline__ int32_t cta_min(int32_t v, int32_t *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = __reduce_min_sync(0xffffffffu, v);
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    x = __reduce_min_sync(0xffffffffu, sm[lane]);
    __syncthreads();
    return x;
}

__device__ __forceinline__ int32_t cta_or(int32_t v, int32_t *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = static_cast<int32_t>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(v)));
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    x = static_cast<int32_t>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(sm[lane])));
    __syncthreads();
    return x;
}

// Steps (1)-(4) for the whole batch, one CTA.  Thread t owns the consecutive
// requests [t * per, (t + 1) * per).
__global__ void __launch_bounds__(kPlanThreads, 1) alloc_plan_kernel(AllocParams p) {
    __shared__ long long sm64[32];
    __shared__ int32_t sm32[32];
    pdl_wait();   // completed_tokens may come from the kernel before
    pdl_trigger();
    const int n = p.n, G = p.G;
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int i0 = min(n, static_cast<int>(threadIdx.x) * per);
    const int i1 = min(n, i0 + per);
    int32_t status = kAllocOk;
    // (1) slots needed, (2) window frees, (3) missing blocks
    for (int i = i0; i < i1; i++) {
        const long long comp = p.completed[p.rows[i]];
        const long long need_len = comp + p.num_new[i] + p.lookahead[i];
        for (int g = 0; g < G; g++) {
            const int have = p.have[g * n + i], lead = p.lead[g * n + i];
            const long long need = (need_len + p.bs[g] - 1) / p.bs[g];
            if (need > p.W[g]) status |= kAllocTooLong;
            int f = 0;
            if (p.window[g] > 0) {
                long long start = comp - (p.window[g] - 1);
                if (start < 0) start = 0;
                const long long to = min(start / p.bs[g], static_cast<long long>(have));
                f = to > lead ? static_cast<int>(to - lead) : 0;
            }
            p.F[g * n + i] = f;
            p.A[g * n + i] = need > have ? static_cast<int>(need - have) : 0;
        }
    }
    // (4) the stack height before each request, and the first refusal
    int first_fail = n;
    for (int g = 0; g < G; g++) {
        long long d = 0;
        for (int i = i0; i < i1; i++) d += p.F[g * n + i] - p.A[g * n + i];
        long long s = p.c0[g] + cta_excl_sum(d, sm64);
        for (int i = i0; i < i1; i++) {
            const int f = p.F[g * n + i], a = p.A[g * n + i];
            p.S[g * n + i] = static_cast<int32_t>(s);
            if (i < first_fail && static_cast<long long>(a) + p.watermark > s + f) first_fail = i;
            s += f - a;
        }
    }
    const int admitted = cta_min(first_fail, sm32);
    const int processed = admitted < n ? admitted + 1 : n;
    // final heights, stack overflow, and for every pusher the lowest height
    // any later processed request starts from
    for (int g = 0; g < G; g++) {
        int32_t top = p.c0[g];
        if (processed > 0) {
            const int last = processed - 1;
            top = p.S[g * n + last] + p.F[g * n + last] - (last < admitted ? p.A[g * n + last] : 0);
        }
        int32_t lo = INT32_MAX;
        const int j1 = min(i1, processed);
        for (int i = i0; i < j1; i++) {
            const long long hi = static_cast<long long>(p.S[g * n + i]) + p.F[g * n + i];
            if (hi > p.cap[g]) status |= kAllocStackFull;
            lo = min(lo, p.S[g * n + i]);
        }
        int32_t cur = cta_suffix_min_excl(lo, top, sm32);
        for (int i = j1 - 1; i >= i0; i--) {
            p.suf[g * n + i] = cur;
            cur = min(cur, p.S[g * n + i]);
        }
        if (threadIdx.x == 0) p.res[8 + g] = top;
    }
    status = cta_or(status, sm32);
    if (threadIdx.x == 0) {
        p.res[0] = status;
        p.res[1] = admitted;
        p.res[2] = processed;
    }
}

// (5) for the admitted requests: each pops A ids; position p = S + F - 1 - k
// goes to table entry have + k.
__global__ void __launch_bounds__(kThreads) alloc_pop_kernel(AllocParams p) {
    pdl_wait();
    pdl_trigger();
    if (p.res[0] != kAllocOk) return;
    const int n = p.n, lane = threadIdx.x & 31;
    const int admitted = p.res[1];
    const long long items = static_cast<long long>(p.G) * n;
    const long long stride = static_cast<long long>(gridDim.x) * kWarps;
    for (long long it = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items;
         it += stride) {
        const int g = static_cast<int>(it / n), i = static_cast<int>(it % n);
        if (i >= admitted) continue;
        const int a = p.A[g * n + i];
        if (a == 0) continue;
        const int S = p.S[g * n + i], f = p.F[g * n + i];
        const int have = p.have[g * n + i], lead = p.lead[g * n + i];
        const int W = p.W[g];
        int32_t *line = p.table[g] + static_cast<long long>(p.rows[i]) * W;
        // own frees (positions S .. S + f - 1), still in the row
        const int own = min(a, f);
        for (int k = lane; k < own; k += 32) line[have + k] = line[lead + f - 1 - k];
        if (a <= f) continue;
        // deeper positions [lo, S): walk back over earlier requests
        const int lo = S + f - a;
        int carry = S;   // positions >= carry are resolved
        for (int base = i - 1; base >= 0 && carry > lo; base -= 32) {
            const int m = base - lane;
            const int Sm = m >= 0 ? p.S[g * n + m] : INT32_MAX;
            int incl = Sm;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl = min(incl, y);
            }
            int excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = INT32_MAX;
            const int pre = min(carry, excl);
            if (m >= 0 && Sm < pre) {
                // request m pushed every position in [Sm, pre) still live here
                const int32_t *src = p.table[g] + static_cast<long long>(p.rows[m]) * W +
                                     p.lead[g * n + m] - Sm;
                for (int q = max(Sm, lo); q < pre; q++) line[have + (S + f - 1 - q)] = src[q];
            }
            carry = min(carry, __shfl_sync(0xffffffffu, incl, 31));
        }
        // positions no earlier request reached: the stack as the call found it
        for (int q = lo + lane; q < carry; q += 32) line[have + (S + f - 1 - q)] = p.pool[g][q];
    }
}

// (2) for the processed requests: push the freed ids that survive in the
// final stack, then clear them from the rows.
__global__ void __launch_bounds__(kThreads) alloc_push_kernel(AllocParams p) {
    pdl_wait();   // the pops read ids these pushes overwrite or clear
    pdl_trigger();
    if (p.res[0] != kAllocOk) return;
    const int n = p.n, lane = threadIdx.x & 31;
    const int processed = p.res[2];
    const long long items = static_cast<long long>(p.G) * n;
    const long long stride = static_cast<long long>(gridDim.x) * kWarps;
    for (long long it = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items;
         it += stride) {
        const int g = static_cast<int>(it / n), j = static_cast<int>(it % n);
        if (j >= processed) continue;
        const int f = p.F[g * n + j];
        if (f == 0) continue;
        const int S = p.S[g * n + j], lead = p.lead[g * n + j], limit = p.suf[g * n + j];
        int32_t *line = p.table[g] + static_cast<long long>(p.rows[j]) * p.W[g];
        for (int k = lane; k < f; k += 32) {
            const int32_t id = line[lead + k];
            if (S + k < limit) p.pool[g][S + k] = id;
            line[lead + k] = -1;
        }
    }
}

int ensure_pool(pkv_state *st, int g) {
    GroupState &gs = st->groups[g];
    if (!gs.d_pool)
        PKV_CUDA_TRY(cudaMalloc(&gs.d_pool, static_cast<size_t>(gs.num_blocks) * 4));
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_pool_reset(pkv_state *st, int32_t group, const int32_t *free_ids, int32_t count,
                   pkv_stream_t stream) {
    if (!st || group < 0 || group >= st->num_groups || count < 0) return PKV_ERR_INVALID_ARG;
    GroupState &gs = st->groups[group];
    if (count > gs.num_blocks || (count > 0 && !free_ids)) return PKV_ERR_INVALID_ARG;
    for (int32_t k = 0; k < count; k++)
        if (free_ids[k] < 0 || free_ids[k] >= gs.num_blocks) return PKV_ERR_INVALID_ARG;
    int rc = ensure_pool(st, group);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = as_stream(stream);
    const int64_t piece = static_cast<int64_t>(stage_limit(st) / 4);
    for (int64_t off = 0; off < count; off += piece) {
        const int64_t m = std::min<int64_t>(piece, count - off);
        int status;
        char *buf = st->ring.reserve(static_cast<size_t>(m) * 4, &status);
        if (!buf) return status;
        memcpy(buf, free_ids + off, static_cast<size_t>(m) * 4);
        PKV_CUDA_TRY(cudaMemcpyAsync(gs.d_pool + off, buf, static_cast<size_t>(m) * 4,
                                     cudaMemcpyHostToDevice, s));
        rc = st->ring.fence(s);
        if (rc != PKV_OK) return rc;
    }
    gs.pool_count = count;
    return PKV_OK;
}

int pkv_pool_size(pkv_state *st, int32_t group, int32_t *count) {
    if (!st || !count || group < 0 || group >= st->num_groups) return PKV_ERR_INVALID_ARG;
    *count = st->groups[group].pool_count;
    return PKV_OK;
}

int pkv_pool_read(pkv_state *st, int32_t group, int32_t *ids, int32_t max_count,
                  pkv_stream_t stream) {
    if (!st || group < 0 || group >= st->num_groups || max_count < 0) return PKV_ERR_INVALID_ARG;
    const GroupState &gs = st->groups[group];
    const int32_t m = std::min(max_count, gs.pool_count);
    if (m > 0 && !ids) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (m > 0)
        PKV_CUDA_TRY(cudaMemcpyAsync(ids, gs.d_pool, static_cast<size_t>(m) * 4,
                                     cudaMemcpyDeviceToHost, s));
    PKV_CUDA_TRY(cudaStreamSynchronize(s));
    return PKV_OK;
}

int pkv_allocate_slots(pkv_state *st, const int32_t *rows, const int32_t *num_new_tokens,
                       const int32_t *num_lookahead, int32_t n, const int32_t *sliding_window,
                       int32_t watermark_blocks, int32_t *out_admitted, int32_t *out_new_blocks,
                       pkv_stream_t stream) {
    if (!st || !out_admitted || n < 0 || n > PKV_MAX_BATCH || watermark_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!rows || !num_new_tokens)) return PKV_ERR_INVALID_ARG;
    const int G = st->num_groups;
    for (int g = 0; g < G; g++) {
        const int rc = ensure_pool(st, g);
        if (rc != PKV_OK) return rc;
        if (sliding_window && sliding_window[g] < 0) return PKV_ERR_INVALID_ARG;
    }
    // ---- validation: live, distinct rows; counts not negative -------------
    if (++st->seen_gen == 0) {
        std::fill(st->seen.begin(), st->seen.end(), 0u);
        std::fill(st->seen2.begin(), st->seen2.end(), 0u);
        st->seen_gen = 1;
    }
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        if (st->seen[r] == st->seen_gen) return PKV_ERR_INVALID_ARG;   // listed twice
        st->seen[r] = st->seen_gen;
        if (num_new_tokens[i] < 0 || (num_lookahead && num_lookahead[i] < 0))
            return PKV_ERR_INVALID_ARG;
    }
    *out_admitted = 0;
    if (n == 0) return PKV_OK;
    // ---- stage: rows, counts, lookahead, held and leading-null blocks ------
    const size_t nn = static_cast<size_t>(n), gn = static_cast<size_t>(G) * nn;
    const size_t in_words = 3 * nn + 2 * gn;
    const size_t words = in_words + 4 * gn + kResWords;
    if (words * 4 > stage_limit(st)) return PKV_ERR_INVALID_ARG;   // state's ring too small
    int status;
    int32_t *h = reinterpret_cast<int32_t *>(st->ring.reserve(in_words * 4, &status));
    if (!h) return status;
    memcpy(h, rows, nn * 4);
    memcpy(h + nn, num_new_tokens, nn * 4);
    if (num_lookahead)
        memcpy(h + 2 * nn, num_lookahead, nn * 4);
    else
        memset(h + 2 * nn, 0, nn * 4);
    for (int g = 0; g < G; g++) {
        const GroupState &gs = st->groups[g];
        int32_t *hv = h + 3 * nn + g * nn, *ld = h + 3 * nn + gn + g * nn;
        for (int32_t i = 0; i < n; i++) {
            hv[i] = gs.nblk[rows[i]];
            ld[i] = gs.lead_null[rows[i]];
        }
    }
    cudaStream_t s = as_stream(stream);
    int32_t *d = reinterpret_cast<int32_t *>(st->d_apply);
    cudaError_t e = cudaMemcpyAsync(d, h, in_words * 4, cudaMemcpyHostToDevice, s);
    int rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    AllocParams p = {};
    p.rows = d;
    p.num_new = d + nn;
    p.lookahead = d + 2 * nn;
    p.have = d + 3 * nn;
    p.lead = d + 3 * nn + gn;
    p.completed = st->d_completed;
    p.S = d + in_words;
    p.suf = p.S + gn;
    p.F = p.suf + gn;
    p.A = p.F + gn;
    p.res = p.A + gn;   // F, A and res are contiguous: one copy back
    p.n = n;
    p.G = G;
    p.watermark = watermark_blocks;
    for (int g = 0; g < G; g++) {
        GroupState &gs = st->groups[g];
        p.bs[g] = gs.block_size;
        p.W[g] = gs.width;
        p.window[g] = sliding_window ? sliding_window[g] : 0;
        p.c0[g] = gs.pool_count;
        p.cap[g] = static_cast<int32_t>(gs.num_blocks);
        p.table[g] = gs.d_table;
        p.pool[g] = gs.d_pool;
    }
    PKV_CUDA_TRY(launch_pdl(alloc_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p));
    const long long warps = static_cast<long long>(G) * n;
    const long long wave = static_cast<long long>(st->num_sms) * (2048 / kThreads);
    const unsigned grid =
        static_cast<unsigned>(std::min<long long>((warps + kWarps - 1) / kWarps, wave));
    PKV_CUDA_TRY(launch_pdl(alloc_pop_kernel, dim3(grid), dim3(kThreads), 0, s, p));
    PKV_CUDA_TRY(launch_pdl(alloc_push_kernel, dim3(grid), dim3(kThreads), 0, s, p));
    // ---- results back (synchronous: the caller needs admission now) --------
    const size_t back = 2 * gn + kResWords;
    int32_t *hb = reinterpret_cast<int32_t *>(st->ring.reserve(back * 4, &status));
    if (!hb) return status;
    e = cudaMemcpyAsync(hb, p.F, back * 4, cudaMemcpyDeviceToHost, s);
    rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    PKV_CUDA_TRY(cudaStreamSynchronize(s));
    const int32_t *hF = hb, *hA = hb + gn, *res = hb + 2 * gn;
    if (res[0] != kAllocOk) return PKV_ERR_CAPACITY;   // nothing was moved
    const int32_t admitted = res[1], processed = res[2];
    for (int g = 0; g < G; g++) {
        GroupState &gs = st->groups[g];
        for (int32_t i = 0; i < admitted; i++) gs.nblk[rows[i]] += hA[g * nn + i];
        for (int32_t i = 0; i < processed; i++) gs.lead_null[rows[i]] += hF[g * nn + i];
        gs.pool_count = res[8 + g];
    }
    if (out_new_blocks)
        for (int32_t i = 0; i < n; i++)
            for (int g = 0; g < G; g++)
                out_new_blocks[static_cast<size_t>(i) * G + g] = i < admitted ? hA[g * nn + i] : 0;
    *out_admitted = admitted;
    return PKV_OK;
}

int pkv_release_blocks(pkv_state *st, const int32_t *rows, int32_t n, pkv_stream_t stream) {
    if (!st || n < 0 || (n > 0 && !rows)) return PKV_ERR_INVALID_ARG;
    const int G = st->num_groups;
    if (++st->seen_gen == 0) {
        std::fill(st->seen.begin(), st->seen.end(), 0u);
        std::fill(st->seen2.begin(), st->seen2.end(), 0u);
        st->seen_gen = 1;
    }
    int32_t add[PKV_MAX_GROUPS] = {0};
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        if (st->seen[r] == st->seen_gen) return PKV_ERR_INVALID_ARG;
        st->seen[r] = st->seen_gen;
        for (int g = 0; g < G; g++) add[g] += st->groups[g].nblk[r] - st->groups[g].lead_null[r];
    }
    for (int g = 0; g < G; g++) {
        const int rc = ensure_pool(st, g);
        if (rc != PKV_OK) return rc;
        if (static_cast<int64_t>(st->groups[g].pool_count) + add[g] > st->groups[g].num_blocks)
            return PKV_ERR_CAPACITY;
    }
    std::vector<MoveOp> pushes;
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            const int32_t from = gs.lead_null[r], to = gs.nblk[r];
            if (to > from) {
                int32_t *row = gs.d_table + static_cast<int64_t>(r) * gs.width;
                pushes.push_back(MoveOp{gs.d_pool + gs.pool_count, row + from, to - from, 1, 1, 0});
                gs.pool_count += to - from;
            }
            gs.nblk[r] = 0;
            gs.lead_null[r] = 0;
        }
    }
    if (pushes.empty()) return PKV_OK;
    return launch_moves(st, pushes, as_stream(stream));
}

}  // extern "C"
