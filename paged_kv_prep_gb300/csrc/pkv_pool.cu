// Free-block pools and allocate_slots.
//
// "allocate_slots()" section of "从源码读 vLLM Scheduler": per request, in
// order -- count the slots needed (computed + new + speculative lookahead),
// free the sliding-window blocks no longer needed, count the new blocks
// actually missing, keep a watermark in reserve and refuse if
// required = new + watermark exceeds available = free - reserved, otherwise
// allocate.  The scheduler stops at a refused request.
//
// GB300 split.  Admission only needs counts, which the host mirrors, so the
// CPU decides it at once (no device round trip) and returns it; the GPU does
// the block-id bookkeeping: ids move from the top of each group's free stack
// into the admitted requests' table rows, and freed sliding-window ids move
// from the rows onto the stack.  Readings (shared with the CPU oracle): one
// call is a batch processed in order; the first refused request and all after
// it are not admitted; the window frees of the requests up to and including
// the refused one go back to the pool after the batch's allocations; the
// stack pops from the top, request after request, and pushes in request order,
// lowest logical block first; blocks wholly before max(0, computed -
// (window - 1)) are out of the window.
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
    if (!st || !out_admitted || n < 0 || watermark_blocks < 0) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!rows || !num_new_tokens)) return PKV_ERR_INVALID_ARG;
    const int G = st->num_groups;
    for (int g = 0; g < G; g++) {
        const int rc = ensure_pool(st, g);
        if (rc != PKV_OK) return rc;
        if (sliding_window && sliding_window[g] < 0) return PKV_ERR_INVALID_ARG;
    }
    // ---- admission (host: counts only) -----------------------------------
    if (++st->seen_gen == 0) {
        std::fill(st->seen.begin(), st->seen.end(), 0u);
        std::fill(st->seen2.begin(), st->seen2.end(), 0u);
        st->seen_gen = 1;
    }
    std::vector<int32_t> newb(static_cast<size_t>(n) * G, 0), fr_from(static_cast<size_t>(n) * G, 0),
        fr_to(static_cast<size_t>(n) * G, 0);
    int32_t taken[PKV_MAX_GROUPS] = {0};
    int32_t admitted = n, processed = n;
    for (int32_t i = 0; i < n; i++) {
        const int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        if (st->seen[r] == st->seen_gen) return PKV_ERR_INVALID_ARG;   // listed twice
        st->seen[r] = st->seen_gen;
        const int32_t la = num_lookahead ? num_lookahead[i] : 0;
        if (num_new_tokens[i] < 0 || la < 0) return PKV_ERR_INVALID_ARG;
        const int64_t need_len = static_cast<int64_t>(st->completed[r]) + num_new_tokens[i] + la;
        bool refused = false;
        for (int g = 0; g < G; g++) {
            const GroupState &gs = st->groups[g];
            const int32_t have = gs.nblk[r];
            const int64_t need = (need_len + gs.block_size - 1) / gs.block_size;
            if (need > gs.width) return PKV_ERR_CAPACITY;
            int32_t from = 0, to = 0;
            if (sliding_window && sliding_window[g] > 0) {
                int64_t start = static_cast<int64_t>(st->completed[r]) - (sliding_window[g] - 1);
                if (start < 0) start = 0;
                to = static_cast<int32_t>(std::min<int64_t>(start / gs.block_size, have));
                from = std::min(gs.lead_null[r], to);
            }
            fr_from[static_cast<size_t>(i) * G + g] = from;
            fr_to[static_cast<size_t>(i) * G + g] = std::max(from, to);
            const int32_t nb = need > have ? static_cast<int32_t>(need - have) : 0;
            newb[static_cast<size_t>(i) * G + g] = nb;
            if (static_cast<int64_t>(nb) + watermark_blocks > gs.pool_count - taken[g]) refused = true;
        }
        if (refused) {
            admitted = i;
            processed = i + 1;
            break;
        }
        for (int g = 0; g < G; g++) taken[g] += newb[static_cast<size_t>(i) * G + g];
    }
    // ---- plan: pops for the admitted, then pushes of the window frees -----
    std::vector<MoveOp> pops, pushes;
    int32_t popped[PKV_MAX_GROUPS] = {0};
    for (int32_t i = 0; i < admitted; i++) {
        const int32_t r = rows[i];
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            const int32_t nb = newb[static_cast<size_t>(i) * G + g];
            if (nb) {
                int32_t *row = gs.d_table + static_cast<int64_t>(r) * gs.width;
                pops.push_back(MoveOp{row + gs.nblk[r], gs.d_pool + (gs.pool_count - 1 - popped[g]),
                                      nb, -1, 0, 0});
                popped[g] += nb;
            }
        }
    }
    int32_t top[PKV_MAX_GROUPS];
    int32_t freed[PKV_MAX_GROUPS] = {0};
    for (int g = 0; g < G; g++) top[g] = st->groups[g].pool_count - popped[g];
    for (int32_t i = 0; i < processed; i++) {
        const int32_t r = rows[i];
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            const int32_t from = fr_from[static_cast<size_t>(i) * G + g];
            const int32_t to = fr_to[static_cast<size_t>(i) * G + g];
            if (to > from) {
                if (static_cast<int64_t>(top[g]) + freed[g] + (to - from) > gs.num_blocks)
                    return PKV_ERR_CAPACITY;   // more ids than the pool holds
                int32_t *row = gs.d_table + static_cast<int64_t>(r) * gs.width;
                pushes.push_back(MoveOp{gs.d_pool + top[g] + freed[g], row + from, to - from, 1, 1, 0});
                freed[g] += to - from;
            }
        }
    }
    cudaStream_t s = as_stream(stream);
    if (!pops.empty()) {
        const int rc = launch_moves(st, pops, s);
        if (rc != PKV_OK) return rc;
    }
    if (!pushes.empty()) {
        const int rc = launch_moves(st, pushes, s);
        if (rc != PKV_OK) return rc;
    }
    // ---- mirrors --------------------------------------------------------------
    for (int32_t i = 0; i < admitted; i++)
        for (int g = 0; g < G; g++) st->groups[g].nblk[rows[i]] += newb[static_cast<size_t>(i) * G + g];
    for (int32_t i = 0; i < processed; i++)
        for (int g = 0; g < G; g++) {
            const int32_t to = fr_to[static_cast<size_t>(i) * G + g];
            if (to > fr_from[static_cast<size_t>(i) * G + g]) st->groups[g].lead_null[rows[i]] = to;
        }
    for (int g = 0; g < G; g++) st->groups[g].pool_count = top[g] + freed[g];
    if (out_new_blocks)
        for (int32_t i = 0; i < n; i++)
            for (int g = 0; g < G; g++)
                out_new_blocks[static_cast<size_t>(i) * G + g] =
                    i < admitted ? newb[static_cast<size_t>(i) * G + g] : 0;
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
