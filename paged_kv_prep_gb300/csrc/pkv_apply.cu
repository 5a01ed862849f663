// One step's scheduler output applied to the request-state table in one go.
//
// "SchedulerOutput" section of "从源码读 vLLM Scheduler": new requests carry
// their full state, cached requests only what changed, finished requests are
// cleaned up; the runner imports the new requests first, then updates the
// block tables of the requests it already has.  Here the finished rows are
// freed first (so new requests can reuse them), then the new requests take
// the lowest free rows ("Design Logic Behind the Dual-Index System", page
// "Deep Dive into vLLM's Scheduling Mechanism"), then the cached requests are
// appended to.
//
// The whole delta is validated against the host mirrors before anything
// changes, turned into a list of int32 copy / fill operations on the device
// table, packed with its payload into the pinned ring, copied to the device
// once and applied by one kernel (one warp per operation).  The operations
// write disjoint memory: a freed row that a new request takes gets no reset
// of its own (the new request rewrites every entry a reset would), and cached
// rows are neither freed nor new.
#include <string.h>

#include <algorithm>
#include <vector>

#include "pkv_async.cuh"
#include "pkv_common.cuh"

namespace {

using namespace pkv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int32_t kOpChunk = 8192;   // ints per operation at most

// dst[0..count) = payload[src..src+count) when src >= 0, else = fill.
struct ApplyOp {
    int32_t *dst;
    int32_t count;
    int32_t src;
    int32_t fill;
    int32_t pad;
};
static_assert(sizeof(ApplyOp) == 24, "ApplyOp layout");

__global__ void __launch_bounds__(kThreads) apply_kernel(const ApplyOp *ops, int32_t nops,
                                                         const int32_t *payload) {
    pdl_wait();   // the table may still be read by the kernel before
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); w < nops;
         w += stride) {
        const ApplyOp op = ops[w];
        if (op.src >= 0) {
            const int32_t *src = payload + op.src;
            for (int32_t i = lane; i < op.count; i += 32) op.dst[i] = src[i];
        } else {
            for (int32_t i = lane; i < op.count; i += 32) op.dst[i] = op.fill;
        }
    }
}

struct Plan {
    std::vector<ApplyOp> ops;
    std::vector<int32_t> payload;

    void copy(int32_t *dst, const int32_t *src, int32_t count) {
        for (int32_t off = 0; off < count; off += kOpChunk) {
            const int32_t m = std::min(kOpChunk, count - off);
            ops.push_back(ApplyOp{dst + off, m, static_cast<int32_t>(payload.size()), 0, 0});
            payload.insert(payload.end(), src + off, src + off + m);
        }
    }
    void fill(int32_t *dst, int32_t value, int32_t count) {
        for (int32_t off = 0; off < count; off += kOpChunk) {
            const int32_t m = std::min(kOpChunk, count - off);
            ops.push_back(ApplyOp{dst + off, m, -1, value, 0});
        }
    }
};

// Stage and launch the plan in pieces that fit the device staging buffer.
int launch_plan(pkv_state *st, Plan &plan, cudaStream_t s) {
    const size_t limit = stage_limit(st);
    size_t a = 0;
    while (a < plan.ops.size()) {
        // take ops [a, b) whose payload is contiguous and fits with them
        size_t b = a;
        int64_t pay_lo = -1, pay_hi = -1;
        size_t bytes = 0;
        while (b < plan.ops.size()) {
            const ApplyOp &op = plan.ops[b];
            int64_t lo = pay_lo, hi = pay_hi;
            if (op.src >= 0) {
                if (lo < 0) lo = op.src;
                hi = static_cast<int64_t>(op.src) + op.count;
            }
            const size_t need = ((b - a + 1) * sizeof(ApplyOp) + 15) / 16 * 16 +
                                static_cast<size_t>(hi > lo && lo >= 0 ? hi - lo : 0) * 4;
            if (need > limit && b > a) break;
            pay_lo = lo;
            pay_hi = hi;
            bytes = need;
            b++;
        }
        const size_t ops_bytes = ((b - a) * sizeof(ApplyOp) + 15) / 16 * 16;
        int status;
        char *buf = st->ring.reserve(bytes, &status);
        if (!buf) return status;
        ApplyOp *ops = reinterpret_cast<ApplyOp *>(buf);
        for (size_t k = a; k < b; k++) {
            ApplyOp op = plan.ops[k];
            if (op.src >= 0) op.src -= static_cast<int32_t>(pay_lo);
            ops[k - a] = op;
        }
        if (pay_lo >= 0)
            memcpy(buf + ops_bytes, plan.payload.data() + pay_lo,
                   static_cast<size_t>(pay_hi - pay_lo) * 4);
        cudaError_t e = cudaMemcpyAsync(st->d_apply, buf, bytes, cudaMemcpyHostToDevice, s);
        const int rc = st->ring.fence(s);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return PKV_ERR_CUDA;
        }
        if (rc != PKV_OK) return rc;
        const int32_t nops = static_cast<int32_t>(b - a);
        const int64_t need = (nops + kWarps - 1) / kWarps;
        const int64_t wave = static_cast<int64_t>(st->num_sms) * (2048 / kThreads);
        const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
        PKV_CUDA_TRY(launch_pdl(apply_kernel, dim3(grid), dim3(kThreads), 0, s,
                                reinterpret_cast<const ApplyOp *>(st->d_apply), nops,
                                reinterpret_cast<const int32_t *>(st->d_apply + ops_bytes)));
        a = b;
    }
    return PKV_OK;
}

bool csr_ok(const int32_t *off, int32_t count) {
    if (!off) return false;
    if (off[0] != 0) return false;
    for (int32_t k = 0; k < count; k++)
        if (off[k + 1] < off[k]) return false;
    return true;
}

}  // namespace

extern "C" int pkv_apply_step(pkv_state *st, const pkv_step_delta *d, int32_t *out_new_rows,
                              pkv_stream_t stream) {
    if (!st || !d) return PKV_ERR_INVALID_ARG;
    if (d->num_finished < 0 || d->num_new < 0 || d->num_cached < 0) return PKV_ERR_INVALID_ARG;
    if (d->num_finished > 0 && !d->finished_rows) return PKV_ERR_INVALID_ARG;
    const int G = st->num_groups;
    // ---- validate ---------------------------------------------------------
    if (++st->seen_gen == 0) {
        std::fill(st->seen.begin(), st->seen.end(), 0u);
        std::fill(st->seen2.begin(), st->seen2.end(), 0u);
        st->seen_gen = 1;
    }
    const uint32_t gen = st->seen_gen;
    for (int32_t f = 0; f < d->num_finished; f++) {
        const int32_t r = d->finished_rows[f];
        if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
        if (!st->active[r]) return PKV_ERR_NOT_ACTIVE;
        if (st->seen[r] == gen) return PKV_ERR_INVALID_ARG;
        st->seen[r] = gen;   // freed in this step
    }
    if (d->num_new > 0) {
        if (!out_new_rows || !d->new_num_computed || !csr_ok(d->new_token_offsets, d->num_new))
            return PKV_ERR_INVALID_ARG;
        if (d->new_token_offsets[d->num_new] > 0 && !d->new_token_ids) return PKV_ERR_INVALID_ARG;
        if (st->pool.size() + static_cast<size_t>(d->num_finished) <
            static_cast<size_t>(d->num_new))
            return PKV_ERR_FULL;
        for (int g = 0; g < G; g++) {
            const int32_t *bo = d->new_block_offsets[g];
            if (!bo) continue;
            if (!csr_ok(bo, d->num_new)) return PKV_ERR_INVALID_ARG;
            if (bo[d->num_new] > 0 && !d->new_block_ids[g]) return PKV_ERR_INVALID_ARG;
        }
        for (int32_t k = 0; k < d->num_new; k++) {
            const int32_t nt = d->new_token_offsets[k + 1] - d->new_token_offsets[k];
            const int32_t nc = d->new_num_computed[k];
            if (nt > st->max_len || nc < 0 || nc > nt) return PKV_ERR_INVALID_ARG;
            for (int g = 0; g < G; g++) {
                const int32_t *bo = d->new_block_offsets[g];
                const int32_t nb = bo ? bo[k + 1] - bo[k] : 0;
                if (nb > st->groups[g].width) return PKV_ERR_INVALID_ARG;
                int32_t lead;
                const int rc = check_block_list(st->groups[g], nb ? d->new_block_ids[g] + bo[k] : nullptr,
                                                nb, true, &lead);
                if (rc != PKV_OK) return rc;
            }
        }
    }
    if (d->num_cached > 0) {
        if (!d->cached_rows || !d->cached_num_computed ||
            !csr_ok(d->cached_token_offsets, d->num_cached))
            return PKV_ERR_INVALID_ARG;
        if (d->cached_token_offsets[d->num_cached] > 0 && !d->cached_token_ids)
            return PKV_ERR_INVALID_ARG;
        for (int g = 0; g < G; g++) {
            const int32_t *bo = d->cached_block_offsets[g];
            if (!bo) continue;
            if (!csr_ok(bo, d->num_cached)) return PKV_ERR_INVALID_ARG;
            if (bo[d->num_cached] > 0 && !d->cached_block_ids[g]) return PKV_ERR_INVALID_ARG;
        }
        for (int32_t c = 0; c < d->num_cached; c++) {
            const int32_t r = d->cached_rows[c];
            if (r < 0 || r >= st->rows) return PKV_ERR_INVALID_ARG;
            if (!st->active[r] || st->seen[r] == gen) return PKV_ERR_NOT_ACTIVE;
            if (st->seen2[r] == gen) return PKV_ERR_INVALID_ARG;   // listed twice
            st->seen2[r] = gen;
            const int32_t k = d->cached_token_offsets[c + 1] - d->cached_token_offsets[c];
            if (static_cast<int64_t>(st->ntok[r]) + k > st->max_len) return PKV_ERR_CAPACITY;
            const int32_t nc = d->cached_num_computed[c];
            if (nc < -1 || nc > st->ntok[r] + k) return PKV_ERR_INVALID_ARG;
            for (int g = 0; g < G; g++) {
                const GroupState &gs = st->groups[g];
                const int32_t *bo = d->cached_block_offsets[g];
                const int32_t m = bo ? bo[c + 1] - bo[c] : 0;
                if (static_cast<int64_t>(gs.nblk[r]) + m > gs.width) return PKV_ERR_CAPACITY;
                int32_t lead;
                const int rc = check_block_list(gs, m ? d->cached_block_ids[g] + bo[c] : nullptr, m,
                                                gs.lead_null[r] == gs.nblk[r], &lead);
                if (rc != PKV_OK) return rc;
            }
        }
    }

    // ---- plan (and update the host mirrors) ---------------------------------
    Plan plan;
    for (int32_t f = 0; f < d->num_finished; f++) {
        const int32_t r = d->finished_rows[f];
        st->active[r] = 0;
        st->completed[r] = 0;
        st->ntok[r] = 0;
        for (int g = 0; g < G; g++) {
            st->groups[g].nblk[r] = 0;
            st->groups[g].lead_null[r] = 0;
        }
        st->pool.push(r);
    }
    for (int32_t k = 0; k < d->num_new; k++) {
        const int32_t r = st->pool.pop();
        out_new_rows[k] = r;
        st->seen[r] = 0;   // reused: the new request rewrites the whole row
        const int32_t t0 = d->new_token_offsets[k];
        const int32_t nt = d->new_token_offsets[k + 1] - t0;
        const int32_t nc = d->new_num_computed[k];
        plan.copy(st->d_completed + r, &nc, 1);
        if (nt) plan.copy(st->d_tokens + static_cast<int64_t>(r) * st->max_len, d->new_token_ids + t0, nt);
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            const int32_t *bo = d->new_block_offsets[g];
            const int32_t nb = bo ? bo[k + 1] - bo[k] : 0;
            int32_t *row = gs.d_table + static_cast<int64_t>(r) * gs.width;
            if (nb) plan.copy(row, d->new_block_ids[g] + bo[k], nb);
            if (gs.width > nb) plan.fill(row + nb, -1, gs.width - nb);
            int32_t lead;
            check_block_list(gs, nb ? d->new_block_ids[g] + bo[k] : nullptr, nb, true, &lead);
            gs.nblk[r] = nb;
            gs.lead_null[r] = lead;
        }
        st->active[r] = 1;
        st->completed[r] = nc;
        st->ntok[r] = nt;
    }
    for (int32_t c = 0; c < d->num_cached; c++) {
        const int32_t r = d->cached_rows[c];
        const int32_t t0 = d->cached_token_offsets[c];
        const int32_t k = d->cached_token_offsets[c + 1] - t0;
        if (k)
            plan.copy(st->d_tokens + static_cast<int64_t>(r) * st->max_len + st->ntok[r],
                      d->cached_token_ids + t0, k);
        st->ntok[r] += k;
        const int32_t nc = d->cached_num_computed[c];
        if (nc >= 0) {
            plan.copy(st->d_completed + r, &nc, 1);
            st->completed[r] = nc;
        }
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            const int32_t *bo = d->cached_block_offsets[g];
            const int32_t m = bo ? bo[c + 1] - bo[c] : 0;
            if (!m) continue;
            plan.copy(gs.d_table + static_cast<int64_t>(r) * gs.width + gs.nblk[r],
                      d->cached_block_ids[g] + bo[c], m);
            int32_t lead;
            check_block_list(gs, d->cached_block_ids[g] + bo[c], m, gs.lead_null[r] == gs.nblk[r],
                             &lead);
            gs.lead_null[r] += lead;
            gs.nblk[r] += m;
        }
    }
    // resets of the freed rows that no new request took
    for (int32_t f = 0; f < d->num_finished; f++) {
        const int32_t r = d->finished_rows[f];
        if (st->seen[r] != gen) continue;
        plan.fill(st->d_completed + r, 0, 1);
        for (int g = 0; g < G; g++) {
            GroupState &gs = st->groups[g];
            plan.fill(gs.d_table + static_cast<int64_t>(r) * gs.width, -1, gs.width);
        }
    }
    if (plan.ops.empty()) return PKV_OK;
    return launch_plan(st, plan, as_stream(stream));
}
