// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <deque>
#include <new>
#include <queue>
#include <vector>

#include "pkv.h"

namespace pkv {

// Thread-local record of the CUDA error behind the last PKV_ERR_CUDA.
void set_cuda_error(cudaError_t e);

#define PKV_CUDA_TRY(expr)                                   \
    do {                                                     \
        cudaError_t e_ = (expr);                             \
        if (e_ != cudaSuccess) {                             \
            ::pkv::set_cuda_error(e_);                       \
            return PKV_ERR_CUDA;                             \
        }                                                    \
    } while (0)

inline cudaStream_t as_stream(pkv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream finishes; it calls pdl_wait()
// before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Pinned host staging ring.  Host inputs are copied here first so that the
// caller may release them as soon as a call returns, and so that the
// host-to-device copies are truly asynchronous.  Each reserved region is
// guarded by an event recorded after the copies that read it; a region is
// only handed out again once its event has completed.
class PinnedRing {
  public:
    int init(size_t bytes);
    void release();
    // Reserve `bytes` (rounded up to 256).  May wait for older copies.
    // Returns nullptr if bytes exceeds the ring.
    char *reserve(size_t bytes, int *status);
    // Record that every region reserved since the last call is read by work
    // enqueued on `s` so far.
    int fence(cudaStream_t s);
    size_t capacity() const { return cap_; }

  private:
    struct Pending {
        size_t begin, end;
        cudaEvent_t ev;
    };
    int wait_front();
    char *base_ = nullptr;
    size_t cap_ = 0;
    size_t head_ = 0;
    size_t unfenced_begin_ = 0;
    bool has_unfenced_ = false;
    std::deque<Pending> pending_;
    std::vector<cudaEvent_t> free_events_;
};

// Rows are handed out lowest-first: a min-heap of free rows.
class RowPool {
  public:
    void init(int32_t rows) {
        free_ = {};
        for (int32_t r = 0; r < rows; r++) free_.push(r);
    }
    bool empty() const { return free_.empty(); }
    size_t size() const { return free_.size(); }
    int32_t pop() {
        int32_t r = free_.top();
        free_.pop();
        return r;
    }
    void push(int32_t r) { free_.push(r); }

  private:
    std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_;
};

struct GroupState {
    int32_t block_size = 0;
    int32_t width = 0;          // W: block-table row length
    int64_t num_blocks = 0;
    int32_t *d_table = nullptr; // [rows][W]
    // host mirrors, per row
    std::vector<int32_t> nblk;       // blocks held
    std::vector<int32_t> lead_null;  // leading -1 entries (freed blocks)
    // free-block stack for pkv_allocate_slots (allocated on first use)
    int32_t *d_pool = nullptr;       // [num_blocks]
    int32_t pool_count = 0;          // host mirror of the stack height
};

}  // namespace pkv

struct pkv_state {
    int device = 0;
    int32_t rows = 0;
    int32_t max_len = 0;
    int32_t num_groups = 0;
    pkv::GroupState groups[PKV_MAX_GROUPS];
    // device tables
    int32_t *d_completed = nullptr;  // [rows]
    int32_t *d_tokens = nullptr;     // [rows][max_len]
    int32_t *d_error = nullptr;      // device error word
    // staging for host arrays of a call, 4 * (PKV_MAX_BATCH + 4) words: a
    // prepare's rows and counts, a block-keys call's rows, offsets and spans
    int32_t *d_sched = nullptr;
    // host mirrors
    std::vector<uint8_t> active;
    std::vector<int32_t> completed;
    std::vector<int32_t> ntok;
    std::vector<uint32_t> seen;      // duplicate-row detection stamps
    std::vector<uint32_t> seen2;     // a second stamp set (pkv_apply_step)
    uint32_t seen_gen = 0;
    char *d_apply = nullptr;         // staging for pkv_apply_step's packed deltas
    // per row, which request of the latest device-schedule call claimed it
    // (call number << 32 | schedule index): finds rows listed twice
    unsigned long long *d_stamp = nullptr;
    uint32_t stamp_gen = 0;
    pkv::RowPool pool;
    pkv::PinnedRing ring;
    int num_sms = 0;
};

namespace pkv {

// Block ids handed to a row: -1 or a pool id, -1 only as a leading run
// (blocks freed out of a sliding window are the oldest ones).  `prefix_open`
// says whether the row so far holds only -1 entries.  Writes the number of
// leading -1 entries of `ids` to *lead_null.
inline int check_block_list(const GroupState &g, const int32_t *ids, int32_t count,
                            bool prefix_open, int32_t *lead_null) {
    int32_t lead = 0;
    bool open = prefix_open;
    for (int32_t j = 0; j < count; j++) {
        const int32_t id = ids[j];
        if (id == -1) {
            if (!open) return PKV_ERR_INVALID_ARG;
            lead++;
        } else {
            if (id < 0 || static_cast<int64_t>(id) >= g.num_blocks) return PKV_ERR_INVALID_ARG;
            open = false;
        }
    }
    *lead_null = lead;
    return PKV_OK;
}

// Bytes of one staged piece (a quarter of the pinned ring).
inline size_t stage_limit(const pkv_state *st) { return st->ring.capacity() / 4; }

// Launch helpers implemented in pkv_prepare.cu.
struct PrepareLaunch {
    const int32_t *d_rows;
    const int32_t *d_counts;
    int32_t n;
    int32_t total_tokens;
    int32_t flags;
    int32_t device_schedule = 0;   // unchecked by the host: detect repeated rows on the GPU
};
int launch_prepare(pkv_state *st, const PrepareLaunch &in, const pkv_batch_out *out,
                   cudaStream_t s);
int launch_advance(pkv_state *st, const int32_t *d_rows, const int32_t *d_counts, int32_t n,
                   cudaStream_t s);

}  // namespace pkv
