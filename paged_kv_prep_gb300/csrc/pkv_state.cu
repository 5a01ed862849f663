// Persistent request-state pool: the worker's per-request table kept in device
// memory, indexed by request_state_index (row), with host mirrors of the
// per-row counters for validation.
//
// Follows "Worker Request State Management" and "Design Logic Behind the
// Dual-Index System" on the page "Deep Dive into vLLM's Scheduling Mechanism:
// The Complete CPU-to-GPU Mapping Pipeline": completed_tokens and the block
// table persist across steps; rows are assigned on arrival and recycled when a
// request completes; add_request initialises a row, update_request appends.
#include <string.h>

#include <algorithm>
#include <new>

#include "pkv_common.cuh"

namespace pkv {

static thread_local int g_last_cuda_error = 0;

void set_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

// ---------------------------------------------------------------------------
// PinnedRing
// ---------------------------------------------------------------------------
int PinnedRing::init(size_t bytes) {
    cap_ = (bytes + 255) & ~size_t(255);
    PKV_CUDA_TRY(cudaHostAlloc(reinterpret_cast<void **>(&base_), cap_, cudaHostAllocDefault));
    head_ = 0;
    return PKV_OK;
}

void PinnedRing::release() {
    for (auto &p : pending_) {
        cudaEventSynchronize(p.ev);
        cudaEventDestroy(p.ev);
    }
    pending_.clear();
    for (auto ev : free_events_) cudaEventDestroy(ev);
    free_events_.clear();
    if (base_) cudaFreeHost(base_);
    base_ = nullptr;
    cap_ = 0;
}

int PinnedRing::wait_front() {
    Pending p = pending_.front();
    pending_.pop_front();
    cudaError_t e = cudaEventSynchronize(p.ev);
    free_events_.push_back(p.ev);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

char *PinnedRing::reserve(size_t bytes, int *status) {
    *status = PKV_OK;
    bytes = std::max<size_t>(256, (bytes + 255) & ~size_t(255));
    if (bytes > cap_) {
        *status = PKV_ERR_INVALID_ARG;
        return nullptr;
    }
    if (head_ + bytes > cap_) {
        // The tail [head_, cap_) is skipped.  Regions still pending there are
        // the oldest ones (front of the queue): retire them before wrapping.
        while (!pending_.empty() && pending_.front().begin >= head_) {
            if ((*status = wait_front()) != PKV_OK) return nullptr;
        }
        head_ = 0;
    }
    // Pending regions overlapping [head_, head_ + bytes) are a prefix of the
    // queue (allocation proceeds forward through the ring).
    while (!pending_.empty()) {
        const Pending &p = pending_.front();
        bool overlap = p.begin < head_ + bytes && head_ < p.end;
        if (!overlap) break;
        if ((*status = wait_front()) != PKV_OK) return nullptr;
    }
    char *ptr = base_ + head_;
    unfenced_begin_ = head_;
    has_unfenced_ = true;
    head_ += bytes;
    return ptr;
}

int PinnedRing::fence(cudaStream_t s) {
    if (!has_unfenced_) return PKV_OK;
    cudaEvent_t ev;
    if (!free_events_.empty()) {
        ev = free_events_.back();
        free_events_.pop_back();
    } else {
        PKV_CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    cudaError_t e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) {
        free_events_.push_back(ev);
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    pending_.push_back(Pending{unfenced_begin_, head_, ev});
    has_unfenced_ = false;
    return PKV_OK;
}

}  // namespace pkv

using pkv::as_stream;
using pkv::check_block_list;
using pkv::stage_limit;

static size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

// Copy `count` int32 from host `src` to device `dst` through the ring.
static int stage_copy(pkv_state *st, int32_t *dst, const int32_t *src, int64_t count,
                      cudaStream_t s) {
    const int64_t piece = static_cast<int64_t>(stage_limit(st) / sizeof(int32_t));
    for (int64_t off = 0; off < count; off += piece) {
        int64_t m = std::min(piece, count - off);
        int status;
        char *buf = st->ring.reserve(static_cast<size_t>(m) * 4, &status);
        if (!buf) return status;
        memcpy(buf, src + off, static_cast<size_t>(m) * 4);
        PKV_CUDA_TRY(cudaMemcpyAsync(dst + off, buf, static_cast<size_t>(m) * 4,
                                     cudaMemcpyHostToDevice, s));
        int rc = st->ring.fence(s);
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

static void free_device(pkv_state *st) {
    cudaFree(st->d_completed);
    cudaFree(st->d_tokens);
    cudaFree(st->d_error);
    cudaFree(st->d_sched);
    cudaFree(st->d_apply);
    cudaFree(st->d_stamp);
    for (int g = 0; g < PKV_MAX_GROUPS; g++) {
        cudaFree(st->groups[g].d_table);
        cudaFree(st->groups[g].d_pool);
    }
    st->ring.release();
}

namespace pkv {
// the prepare path's host-schedule staging (stream, events, buffers) of a
// state, defined in pkv_prepare.cu
void release_prepare_staging(const pkv_state *st);
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 100; }

int pkv_last_cuda_error(void) { return pkv::g_last_cuda_error; }

int pkv_state_create(pkv_state **out, int32_t max_reqs, int32_t max_model_len,
                     int32_t num_groups, const pkv_group_spec *groups, int64_t ring_bytes,
                     pkv_stream_t stream) {
    if (!out || !groups) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_reqs < 1 || max_reqs > 65536 || max_model_len < 1) return PKV_ERR_INVALID_ARG;
    if (num_groups < 1 || num_groups > PKV_MAX_GROUPS) return PKV_ERR_INVALID_ARG;
    if (ring_bytes < 0) return PKV_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; g++) {
        const pkv_group_spec &gs = groups[g];
        if (gs.block_size < 1 || gs.max_blocks_per_req < 1 || gs.num_blocks < 1)
            return PKV_ERR_INVALID_ARG;
        // slot ids must fit comfortably in int64 and block ids in int32
        if (gs.num_blocks > INT32_MAX) return PKV_ERR_INVALID_ARG;
    }
    cudaStream_t s = as_stream(stream);
    pkv_state *st = new (std::nothrow) pkv_state();
    if (!st) return PKV_ERR_INVALID_ARG;
    st->rows = max_reqs;
    st->max_len = max_model_len;
    st->num_groups = num_groups;

    int rc = PKV_OK;
    auto fail = [&](int code) {
        free_device(st);
        delete st;
        return code;
    };
    cudaError_t e = cudaGetDevice(&st->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&st->num_sms, cudaDevAttrMultiProcessorCount, st->device);
    const size_t rows = static_cast<size_t>(max_reqs);
    if (e == cudaSuccess) e = cudaMalloc(&st->d_completed, rows * 4);
    if (e == cudaSuccess) e = cudaMalloc(&st->d_tokens, rows * static_cast<size_t>(max_model_len) * 4);
    if (e == cudaSuccess) e = cudaMalloc(&st->d_error, 256);
    if (e == cudaSuccess) e = cudaMalloc(&st->d_stamp, rows * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemsetAsync(st->d_stamp, 0, rows * sizeof(unsigned long long), s);
    // staged per-call host arrays, each starting 16-byte aligned: the
    // schedule's rows and counts, or pkv_block_keys' rows, offsets and long
    // requests (at most three arrays of up to PKV_MAX_BATCH + 1 entries)
    if (e == cudaSuccess) e = cudaMalloc(&st->d_sched, 4 * (PKV_MAX_BATCH + 4) * sizeof(int32_t));
    for (int g = 0; g < num_groups && e == cudaSuccess; g++) {
        pkv::GroupState &gs = st->groups[g];
        gs.block_size = groups[g].block_size;
        gs.width = groups[g].max_blocks_per_req;
        gs.num_blocks = groups[g].num_blocks;
        e = cudaMalloc(&gs.d_table, rows * static_cast<size_t>(gs.width) * 4);
        if (e == cudaSuccess) e = cudaMemsetAsync(gs.d_table, 0xFF, rows * gs.width * 4, s);
        gs.nblk.assign(rows, 0);
        gs.lead_null.assign(rows, 0);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(st->d_completed, 0, rows * 4, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(st->d_tokens, 0, rows * static_cast<size_t>(max_model_len) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->d_error, 0, 256, s);
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return fail(PKV_ERR_CUDA);
    }
    rc = st->ring.init(ring_bytes ? static_cast<size_t>(ring_bytes) : (size_t(64) << 20));
    if (rc != PKV_OK) return fail(rc);
    e = cudaMalloc(&st->d_apply, stage_limit(st));
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return fail(PKV_ERR_CUDA);
    }
    st->active.assign(rows, 0);
    st->completed.assign(rows, 0);
    st->ntok.assign(rows, 0);
    st->seen.assign(rows, 0);
    st->seen2.assign(rows, 0);
    st->pool.init(max_reqs);
    *out = st;
    return PKV_OK;
}

int pkv_state_destroy(pkv_state *st) {
    if (!st) return PKV_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    pkv::release_prepare_staging(st);
    free_device(st);
    delete st;
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

int pkv_add_request(pkv_state *st, const int32_t *token_ids, int32_t n_tokens,
                    int32_t num_computed_tokens, const int32_t *const *block_ids,
                    const int32_t *n_blocks, int32_t *out_row, pkv_stream_t stream) {
    if (!st || !out_row || !n_blocks) return PKV_ERR_INVALID_ARG;
    if (n_tokens < 0 || n_tokens > st->max_len) return PKV_ERR_INVALID_ARG;
    if (n_tokens > 0 && !token_ids) return PKV_ERR_INVALID_ARG;
    if (num_computed_tokens < 0 || num_computed_tokens > n_tokens) return PKV_ERR_INVALID_ARG;
    int32_t lead[PKV_MAX_GROUPS];
    for (int g = 0; g < st->num_groups; g++) {
        const pkv::GroupState &gs = st->groups[g];
        if (n_blocks[g] < 0 || n_blocks[g] > gs.width) return PKV_ERR_INVALID_ARG;
        if (n_blocks[g] > 0 && (!block_ids || !block_ids[g])) return PKV_ERR_INVALID_ARG;
        int rc = check_block_list(gs, n_blocks[g] ? block_ids[g] : nullptr, n_blocks[g], true,
                                  &lead[g]);
        if (rc != PKV_OK) return rc;
    }
    if (st->pool.empty()) return PKV_ERR_FULL;
    cudaStream_t s = as_stream(stream);

    // One staging region: completed, then each group's full table row
    // (ids followed by -1, which also clears what a previous tenant left).
    size_t bytes = 16;
    for (int g = 0; g < st->num_groups; g++) bytes += round16(st->groups[g].width * 4);
    if (bytes > stage_limit(st)) return PKV_ERR_INVALID_ARG;
    int status;
    char *buf = st->ring.reserve(bytes, &status);
    if (!buf) return status;
    const int32_t row = st->pool.pop();
    auto undo = [&](int code) {
        st->pool.push(row);
        return code;
    };
    memcpy(buf, &num_computed_tokens, 4);
    size_t off = 16;
    cudaError_t e = cudaMemcpyAsync(st->d_completed + row, buf, 4, cudaMemcpyHostToDevice, s);
    for (int g = 0; g < st->num_groups && e == cudaSuccess; g++) {
        pkv::GroupState &gs = st->groups[g];
        int32_t *line = reinterpret_cast<int32_t *>(buf + off);
        if (n_blocks[g]) memcpy(line, block_ids[g], static_cast<size_t>(n_blocks[g]) * 4);
        for (int32_t j = n_blocks[g]; j < gs.width; j++) line[j] = -1;
        e = cudaMemcpyAsync(gs.d_table + static_cast<int64_t>(row) * gs.width, line,
                            static_cast<size_t>(gs.width) * 4, cudaMemcpyHostToDevice, s);
        off += round16(gs.width * 4);
    }
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        st->ring.fence(s);
        return undo(PKV_ERR_CUDA);
    }
    int rc = st->ring.fence(s);
    if (rc != PKV_OK) return undo(rc);
    rc = stage_copy(st, st->d_tokens + static_cast<int64_t>(row) * st->max_len, token_ids,
                    n_tokens, s);
    if (rc != PKV_OK) return undo(rc);

    st->active[row] = 1;
    st->completed[row] = num_computed_tokens;
    st->ntok[row] = n_tokens;
    for (int g = 0; g < st->num_groups; g++) {
        st->groups[g].nblk[row] = n_blocks[g];
        st->groups[g].lead_null[row] = lead[g];
    }
    *out_row = row;
    return PKV_OK;
}

int pkv_update_request(pkv_state *st, int32_t row, const int32_t *const *new_block_ids,
                       const int32_t *n_new_blocks, const int32_t *new_token_ids,
                       int32_t n_new_tokens, int32_t num_computed_tokens, pkv_stream_t stream) {
    if (!st || row < 0 || row >= st->rows) return PKV_ERR_INVALID_ARG;
    if (!st->active[row]) return PKV_ERR_NOT_ACTIVE;
    if (n_new_tokens < 0 || (n_new_tokens > 0 && !new_token_ids)) return PKV_ERR_INVALID_ARG;
    if (num_computed_tokens < -1) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(st->ntok[row]) + n_new_tokens > st->max_len) return PKV_ERR_CAPACITY;
    const int32_t new_ntok = st->ntok[row] + n_new_tokens;
    if (num_computed_tokens > new_ntok) return PKV_ERR_INVALID_ARG;
    int32_t lead[PKV_MAX_GROUPS];
    int32_t add[PKV_MAX_GROUPS];
    for (int g = 0; g < st->num_groups; g++) {
        const pkv::GroupState &gs = st->groups[g];
        add[g] = n_new_blocks ? n_new_blocks[g] : 0;
        if (add[g] < 0) return PKV_ERR_INVALID_ARG;
        if (add[g] > 0 && (!new_block_ids || !new_block_ids[g])) return PKV_ERR_INVALID_ARG;
        if (static_cast<int64_t>(gs.nblk[row]) + add[g] > gs.width) return PKV_ERR_CAPACITY;
        const bool open = gs.lead_null[row] == gs.nblk[row];
        int rc = check_block_list(gs, add[g] ? new_block_ids[g] : nullptr, add[g], open, &lead[g]);
        if (rc != PKV_OK) return rc;
    }
    cudaStream_t s = as_stream(stream);
    size_t bytes = 16;
    for (int g = 0; g < st->num_groups; g++) bytes += round16(static_cast<size_t>(add[g]) * 4);
    if (bytes > stage_limit(st)) return PKV_ERR_INVALID_ARG;
    int status;
    char *buf = st->ring.reserve(bytes, &status);
    if (!buf) return status;
    cudaError_t e = cudaSuccess;
    if (num_computed_tokens >= 0) {
        memcpy(buf, &num_computed_tokens, 4);
        e = cudaMemcpyAsync(st->d_completed + row, buf, 4, cudaMemcpyHostToDevice, s);
    }
    size_t off = 16;
    for (int g = 0; g < st->num_groups && e == cudaSuccess; g++) {
        if (!add[g]) continue;
        pkv::GroupState &gs = st->groups[g];
        memcpy(buf + off, new_block_ids[g], static_cast<size_t>(add[g]) * 4);
        e = cudaMemcpyAsync(gs.d_table + static_cast<int64_t>(row) * gs.width + gs.nblk[row],
                            buf + off, static_cast<size_t>(add[g]) * 4, cudaMemcpyHostToDevice, s);
        off += round16(static_cast<size_t>(add[g]) * 4);
    }
    int rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    rc = stage_copy(st, st->d_tokens + static_cast<int64_t>(row) * st->max_len + st->ntok[row],
                    new_token_ids, n_new_tokens, s);
    if (rc != PKV_OK) return rc;
    st->ntok[row] = new_ntok;
    if (num_computed_tokens >= 0) st->completed[row] = num_computed_tokens;
    for (int g = 0; g < st->num_groups; g++) {
        pkv::GroupState &gs = st->groups[g];
        gs.lead_null[row] += lead[g];
        gs.nblk[row] += add[g];
    }
    return PKV_OK;
}

int pkv_remove_request(pkv_state *st, int32_t row, pkv_stream_t stream) {
    if (!st || row < 0 || row >= st->rows) return PKV_ERR_INVALID_ARG;
    if (!st->active[row]) return PKV_ERR_NOT_ACTIVE;
    cudaStream_t s = as_stream(stream);
    PKV_CUDA_TRY(cudaMemsetAsync(st->d_completed + row, 0, 4, s));
    for (int g = 0; g < st->num_groups; g++) {
        pkv::GroupState &gs = st->groups[g];
        PKV_CUDA_TRY(cudaMemsetAsync(gs.d_table + static_cast<int64_t>(row) * gs.width, 0xFF,
                                     static_cast<size_t>(gs.width) * 4, s));
        gs.nblk[row] = 0;
        gs.lead_null[row] = 0;
    }
    st->active[row] = 0;
    st->completed[row] = 0;
    st->ntok[row] = 0;
    st->pool.push(row);
    return PKV_OK;
}

int pkv_row_info(pkv_state *st, int32_t row, int32_t *active, int32_t *completed,
                 int32_t *n_tokens, int32_t *n_blocks) {
    if (!st || row < 0 || row >= st->rows) return PKV_ERR_INVALID_ARG;
    if (active) *active = st->active[row];
    if (completed) *completed = st->completed[row];
    if (n_tokens) *n_tokens = st->ntok[row];
    if (n_blocks)
        for (int g = 0; g < st->num_groups; g++) n_blocks[g] = st->groups[g].nblk[row];
    return PKV_OK;
}

int pkv_read_row(pkv_state *st, int32_t row, int32_t *completed, int32_t *tokens,
                 int32_t n_tokens, int32_t *const *block_table, pkv_stream_t stream) {
    if (!st || row < 0 || row >= st->rows) return PKV_ERR_INVALID_ARG;
    if (n_tokens < 0 || n_tokens > st->max_len || (n_tokens > 0 && !tokens))
        return PKV_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (completed)
        PKV_CUDA_TRY(cudaMemcpyAsync(completed, st->d_completed + row, 4, cudaMemcpyDeviceToHost, s));
    if (n_tokens)
        PKV_CUDA_TRY(cudaMemcpyAsync(tokens, st->d_tokens + static_cast<int64_t>(row) * st->max_len,
                                     static_cast<size_t>(n_tokens) * 4, cudaMemcpyDeviceToHost, s));
    for (int g = 0; block_table && g < st->num_groups; g++) {
        if (!block_table[g]) continue;
        pkv::GroupState &gs = st->groups[g];
        PKV_CUDA_TRY(cudaMemcpyAsync(block_table[g], gs.d_table + static_cast<int64_t>(row) * gs.width,
                                     static_cast<size_t>(gs.width) * 4, cudaMemcpyDeviceToHost, s));
    }
    PKV_CUDA_TRY(cudaStreamSynchronize(s));
    return PKV_OK;
}

int pkv_get_error(pkv_state *st, int32_t *code) {
    if (!st || !code) return PKV_ERR_INVALID_ARG;
    PKV_CUDA_TRY(cudaDeviceSynchronize());
    PKV_CUDA_TRY(cudaMemcpy(code, st->d_error, 4, cudaMemcpyDeviceToHost));
    PKV_CUDA_TRY(cudaMemset(st->d_error, 0, 4));
    PKV_CUDA_TRY(cudaDeviceSynchronize());
    return PKV_OK;
}

int pkv_state_error_word(pkv_state *st, int32_t **d_error) {
    if (!st || !d_error) return PKV_ERR_INVALID_ARG;
    *d_error = st->d_error;
    return PKV_OK;
}

}  // extern "C"
