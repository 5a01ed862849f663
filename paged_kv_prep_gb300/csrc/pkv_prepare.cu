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
//   * every CTA stages the n scheduled counts in shared memory and scans them
//     (warp-shuffle scan) in schedule order;
//   * the whole step is one flat space of work units, request i owning
//     alpha + n_i consecutive units (alpha 16-byte chunks of its block-table
//     rows, then one unit per token); each CTA takes an equal contiguous slice
//     of that space, so the grid is balanced whatever the mix of decodes and
//     long prefill chunks, and is sized to the SM count;
//   * a CTA needs each of its requests' batch rank and query_start_loc, i.e.
//     the request's place in the stable sort and the sum of the counts that
//     precede it.  One warp gets both for one request by comparing its count
//     with every count in shared memory ((n_j, j) < (n_i, i)) and reducing --
//     no grid-wide barrier and no second kernel;
//   * the block-table rows move as 16-byte vectors with several loads in
//     flight per thread before the stores; token units write positions,
//     input_ids and one int64 slot per group with coalesced accesses.
#include <limits.h>

#include "pkv_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = kWarps;      // requests ranked per round, one per warp
constexpr int kUnroll = 4;          // loads in flight per thread per round
constexpr int64_t kMinUnitsPerCta = 2048;

struct PrepParams {
    const int32_t *rows;        // [n] request_state_index per scheduled request
    const int32_t *counts;      // [n] num_scheduled_tokens
    int32_t n;
    int32_t T;
    int32_t counts_aligned;     // counts is 16-byte aligned
    int32_t num_rows;
    int32_t max_len;
    int32_t G;
    int32_t vec;                // block-table rows move as 16-byte chunks
    int64_t tok_stride;
    const int32_t *completed;
    const int32_t *tokens;
    int64_t alpha;              // gather units per request (sum over groups)
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

// Block-wide exclusive scan of one int64 per thread; returns the prefix and
// writes the block total to *total.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_tot,
                                                        int64_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int64_t o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int d = 1; d < kWarps; d <<= 1) {
            int64_t o = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += o;
        }
        if (lane < kWarps) warp_tot[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    const int64_t before = warp ? warp_tot[warp - 1] : 0;
    *total = warp_tot[kWarps - 1];
    return before + inc - v;
}

__global__ void __launch_bounds__(kThreads) prepare_kernel(const PrepParams p) {
    extern __shared__ __align__(16) int32_t smem[];
    const int n = p.n;
    const int n4 = (n + 3) & ~3;
    int32_t *s_cnt = smem;        // [n4] counts (padding = INT_MAX, never precedes)
    int32_t *s_U = smem + n4;     // [n + 1] schedule-order exclusive prefix

    __shared__ int64_t s_warp_tot[kWarps];
    __shared__ int64_t s_C[kBatch + 1];
    __shared__ int32_t s_rank[kBatch], s_start[kBatch], s_row[kBatch], s_comp[kBatch];
    __shared__ int32_t s_cnt_b[kBatch], s_ok[kBatch];
    __shared__ int32_t s_ga[kBatch], s_gpre[kBatch + 1], s_ka[kBatch], s_tpre[kBatch + 1];
    __shared__ int32_t s_nreq;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- 1. stage the counts ------------------------------------------------
    int bad = 0;
    if (p.counts_aligned) {
        const int4 *src = reinterpret_cast<const int4 *>(p.counts);
        int4 *dst = reinterpret_cast<int4 *>(s_cnt);
        for (int j4 = tid; j4 < n / 4; j4 += kThreads) {
            int4 c = ld_stream(src + j4);
            bad |= (c.x < 1) | (c.y < 1) | (c.z < 1) | (c.w < 1);
            dst[j4] = c;
        }
        for (int j = (n / 4) * 4 + tid; j < n4; j += kThreads) {
            int32_t c = j < n ? ld_stream(p.counts + j) : INT_MAX;
            bad |= (j < n) & (c < 1);
            s_cnt[j] = c;
        }
    } else {
        for (int j = tid; j < n4; j += kThreads) {
            int32_t c = j < n ? ld_stream(p.counts + j) : INT_MAX;
            bad |= (j < n) & (c < 1);
            s_cnt[j] = c;
        }
    }
    __syncthreads();

    // ---- 2. schedule-order exclusive scan (each thread a contiguous run) ----
    const int seg = (n + kThreads - 1) / kThreads;
    const int b0 = min(tid * seg, n), b1 = min(b0 + seg, n);
    int64_t run = 0;
    for (int j = b0; j < b1; j++) run += s_cnt[j];
    int64_t total;
    int64_t base = block_exclusive_scan(run, s_warp_tot, &total);
    bad = __syncthreads_or(bad | (total != p.T));
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) flag(p.err, PKV_DEVERR_COUNT);
        return;
    }
    // every prefix is <= T < 2^31 from here on
    for (int j = b0; j < b1; j++) {
        s_U[j] = static_cast<int32_t>(base);
        base += s_cnt[j];
    }
    if (tid == 0) s_U[n] = p.T;
    __syncthreads();

    // ---- 3. this CTA's slice of the unit space -------------------------------
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * p.units_per_cta;
    const int64_t hi = min(lo + p.units_per_cta, p.total_units);
    if (lo >= hi) return;
    auto C = [&](int i) -> int64_t { return p.alpha * i + s_U[i]; };
    // first request whose units reach lo: largest i with C(i) <= lo
    int l = 0, r = n;
    while (r - l > 1) {
        int m = (l + r) >> 1;
        if (C(m) <= lo) l = m; else r = m;
    }

    const int4 *cnt4 = reinterpret_cast<const int4 *>(s_cnt);
    for (int ib = l; ib < n && C(ib) < hi; ib += kBatch) {
        if (tid == 0) {
            int k = min(kBatch, n - ib);
            while (k > 1 && C(ib + k - 1) >= hi) k--;
            s_nreq = k;
        }
        __syncthreads();
        const int nreq = s_nreq;

        // ---- 4. rank + query_start_loc, one warp per request ----------------
        if (warp < nreq) {
            const int i = ib + warp;
            const int32_t ci = s_cnt[i];
            int32_t row = 0;
            if (lane == 0) row = p.rows[i];
            int32_t cnt = 0, sum = 0;
            for (int j4 = lane; j4 < n4 / 4; j4 += 32) {
                const int4 c = cnt4[j4];
                const int j = j4 * 4;
                const bool a0 = c.x < ci || (c.x == ci && j + 0 < i);
                const bool a1 = c.y < ci || (c.y == ci && j + 1 < i);
                const bool a2 = c.z < ci || (c.z == ci && j + 2 < i);
                const bool a3 = c.w < ci || (c.w == ci && j + 3 < i);
                cnt += a0 + a1 + a2 + a3;
                sum += (a0 ? c.x : 0) + (a1 ? c.y : 0) + (a2 ? c.z : 0) + (a3 ? c.w : 0);
            }
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            sum = __reduce_add_sync(0xffffffffu, sum);
            if (lane == 0) {
                const bool ok = row >= 0 && row < p.num_rows;
                s_rank[warp] = cnt;
                s_start[warp] = sum;
                s_row[warp] = row;
                s_cnt_b[warp] = ci;
                s_ok[warp] = ok;
                s_comp[warp] = ok ? p.completed[row] : 0;
                if (!ok) flag(p.err, PKV_DEVERR_ROW);
            }
        }
        if (tid <= nreq) s_C[tid] = C(ib + tid);
        __syncthreads();

        // ---- 5. per-request scalars, by the CTA that owns the first unit ----
        if (tid == 0) {
            int32_t gp = 0, tp = 0;
            for (int q = 0; q < nreq; q++) {
                const int64_t c0 = s_C[q];
                const int64_t g_lo = max(lo, c0) - c0, g_hi = min(hi, c0 + p.alpha) - c0;
                const int32_t gcount = g_hi > g_lo ? static_cast<int32_t>(g_hi - g_lo) : 0;
                s_ga[q] = static_cast<int32_t>(g_lo);
                s_gpre[q] = gp;
                gp += gcount;
                const int64_t t0 = c0 + p.alpha;
                const int64_t k_lo = max(lo, t0) - t0, k_hi = min(hi, t0 + s_cnt_b[q]) - t0;
                const int32_t tcount = k_hi > k_lo ? static_cast<int32_t>(k_hi - k_lo) : 0;
                s_ka[q] = static_cast<int32_t>(k_lo > 0 ? k_lo : 0);
                s_tpre[q] = tp;
                tp += tcount;
            }
            s_gpre[nreq] = gp;
            s_tpre[nreq] = tp;
        }
        if (tid < nreq && s_C[tid] >= lo) {
            const int32_t rank = s_rank[tid];
            const bool ok = s_ok[tid];
            p.index_mapping[rank] = ok ? s_row[tid] : -1;
            p.qsl[rank] = s_start[tid];
            p.seq_lens[rank] = ok ? s_comp[tid] + s_cnt_b[tid] : -1;
            if (rank == n - 1) p.qsl[n] = s_start[tid] + s_cnt_b[tid];
        }
        __syncthreads();

        // ---- 6. block-table row gather --------------------------------------
        const int32_t gtotal = s_gpre[nreq];
        for (int32_t f0 = 0; f0 < gtotal; f0 += kThreads * kUnroll) {
            if (p.vec) {
                int4 v[kUnroll];
                int4 *dst[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    const int32_t f = f0 + u * kThreads + tid;
                    dst[u] = nullptr;
                    if (f < gtotal) {
                        int q = 0;
                        while (q + 1 < nreq && s_gpre[q + 1] <= f) q++;
                        const int32_t chunk = s_ga[q] + (f - s_gpre[q]);
                        int g = 0;
                        while (chunk >= p.chunk_off[g + 1]) g++;
                        const int32_t e = chunk - p.chunk_off[g];
                        const int64_t w = p.width[g];
                        dst[u] = reinterpret_cast<int4 *>(p.out_table[g] + s_rank[q] * w) + e;
                        v[u] = s_ok[q]
                                   ? ld_stream(reinterpret_cast<const int4 *>(
                                                   p.table[g] + s_row[q] * w) + e)
                                   : make_int4(-1, -1, -1, -1);
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++)
                    if (dst[u]) *dst[u] = v[u];
            } else {
                int32_t v[kUnroll];
                int32_t *dst[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    const int32_t f = f0 + u * kThreads + tid;
                    dst[u] = nullptr;
                    if (f < gtotal) {
                        int q = 0;
                        while (q + 1 < nreq && s_gpre[q + 1] <= f) q++;
                        const int32_t e0 = s_ga[q] + (f - s_gpre[q]);
                        int g = 0;
                        while (e0 >= p.chunk_off[g + 1]) g++;
                        const int32_t e = e0 - p.chunk_off[g];
                        const int64_t w = p.width[g];
                        dst[u] = p.out_table[g] + s_rank[q] * w + e;
                        v[u] = s_ok[q] ? ld_stream(p.table[g] + s_row[q] * w + e) : -1;
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++)
                    if (dst[u]) *dst[u] = v[u];
            }
        }

        // ---- 7. per-token expansion ------------------------------------------
        const int32_t ttotal = s_tpre[nreq];
        for (int32_t f = tid; f < ttotal; f += kThreads) {
            int q = 0;
            while (q + 1 < nreq && s_tpre[q + 1] <= f) q++;
            const int32_t k = s_ka[q] + (f - s_tpre[q]);
            const int32_t t = s_start[q] + k;
            const int32_t pos = s_comp[q] + k;
            const int32_t row = s_row[q];
            bool ok = s_ok[q];
            if (ok && pos >= p.max_len) {
                flag(p.err, PKV_DEVERR_POSITION);
                ok = false;
            }
            p.positions[t] = ok ? pos : -1;
            p.input_ids[t] = ok ? p.tokens[row * p.tok_stride + pos] : -1;
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
        }
        __syncthreads();
    }
}

__global__ void advance_kernel(const int32_t *rows, const int32_t *counts, int32_t n,
                               int32_t num_rows, int32_t *completed) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const int32_t r = rows[i];
        if (r >= 0 && r < num_rows) completed[r] += counts[i];
    }
}

size_t prepare_smem_bytes(int32_t n) {
    const int32_t n4 = (n + 3) & ~3;
    return static_cast<size_t>(n4 + n + 1) * sizeof(int32_t);
}

int ensure_kernel_attributes(int device) {
    static int configured[64] = {0};
    if (device < 0 || device >= 64) return PKV_ERR_INVALID_ARG;
    if (!configured[device]) {
        PKV_CUDA_TRY(cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(prepare_smem_bytes(PKV_MAX_BATCH))));
        configured[device] = 1;
    }
    return PKV_OK;
}

}  // namespace

namespace pkv {

int launch_prepare(pkv_state *st, const PrepareLaunch &in, const pkv_batch_out *out,
                   cudaStream_t s) {
    int rc = ensure_kernel_attributes(st->device);
    if (rc != PKV_OK) return rc;
    PrepParams p = {};
    p.rows = in.d_rows;
    p.counts = in.d_counts;
    p.n = in.n;
    p.T = in.total_tokens;
    p.counts_aligned = (reinterpret_cast<uintptr_t>(in.d_counts) & 15) == 0;
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
    // 16-byte chunks when every table row (state and output) starts 16-byte aligned
    int vec = 1;
    for (int g = 0; g < st->num_groups; g++) {
        const GroupState &gs = st->groups[g];
        if (gs.width % 4 != 0 || (reinterpret_cast<uintptr_t>(out->block_tables[g]) & 15)) vec = 0;
    }
    p.vec = vec;
    int64_t alpha = 0;
    p.chunk_off[0] = 0;
    for (int g = 0; g < st->num_groups; g++) {
        const GroupState &gs = st->groups[g];
        const int32_t units = vec ? gs.width / 4 : gs.width;
        p.chunk_off[g + 1] = p.chunk_off[g] + units;
        p.width[g] = gs.width;
        p.bs[g] = gs.block_size;
        int sh = -1;
        if ((gs.block_size & (gs.block_size - 1)) == 0) {
            sh = 0;
            while ((1 << sh) < gs.block_size) sh++;
        }
        p.bs_shift[g] = sh;
        p.num_blocks[g] = gs.num_blocks;
        p.table[g] = gs.d_table;
        p.out_table[g] = out->block_tables[g];
        p.slots[g] = out->slot_mapping[g];
        alpha += units;
    }
    for (int g = st->num_groups; g < PKV_MAX_GROUPS; g++) p.chunk_off[g + 1] = p.chunk_off[g];
    p.alpha = alpha;
    p.total_units = alpha * in.n + in.total_tokens;

    const size_t smem = prepare_smem_bytes(in.n);
    int per_sm = 0;
    PKV_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prepare_kernel, kThreads,
                                                               smem));
    if (per_sm < 1) per_sm = 1;
    const int64_t max_ctas = static_cast<int64_t>(st->num_sms) * per_sm;
    int64_t per_cta = (p.total_units + max_ctas - 1) / max_ctas;
    if (per_cta < kMinUnitsPerCta) per_cta = kMinUnitsPerCta;
    p.units_per_cta = per_cta;
    const int64_t grid = (p.total_units + per_cta - 1) / per_cta;
    prepare_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    PKV_CUDA_TRY(cudaGetLastError());
    return PKV_OK;
}

int launch_advance(pkv_state *st, const int32_t *d_rows, const int32_t *d_counts, int32_t n,
                   cudaStream_t s) {
    advance_kernel<<<(n + 255) / 256, 256, 0, s>>>(d_rows, d_counts, n, st->rows, st->d_completed);
    PKV_CUDA_TRY(cudaGetLastError());
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
    if (flags & ~PKV_ADVANCE) return PKV_ERR_INVALID_ARG;
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
    if (T > INT32_MAX) return PKV_ERR_INVALID_ARG;
    if (!outputs_ok(st, out, n, T)) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = pkv::as_stream(stream);
    if (n == 0) {
        PKV_CUDA_TRY(cudaMemsetAsync(out->query_start_loc, 0, sizeof(int32_t), s));
        *out_total_tokens = 0;
        return PKV_OK;
    }
    // one host-to-device copy: rows, then counts at a 16-byte aligned offset
    const int32_t n4 = (n + 3) & ~3;
    int status;
    char *buf = st->ring.reserve(static_cast<size_t>(n4 + n) * 4, &status);
    if (!buf) return status;
    memcpy(buf, rows, static_cast<size_t>(n) * 4);
    memcpy(buf + static_cast<size_t>(n4) * 4, num_sched, static_cast<size_t>(n) * 4);
    cudaError_t e = cudaMemcpyAsync(st->d_sched, buf, static_cast<size_t>(n4 + n) * 4,
                                    cudaMemcpyHostToDevice, s);
    int rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        pkv::set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    pkv::PrepareLaunch in{st->d_sched, st->d_sched + n4, n, static_cast<int32_t>(T)};
    rc = pkv::launch_prepare(st, in, out, s);
    if (rc != PKV_OK) return rc;
    if (flags & PKV_ADVANCE) {
        rc = pkv::launch_advance(st, in.d_rows, in.d_counts, n, s);
        if (rc != PKV_OK) return rc;
        for (int32_t i = 0; i < n; i++) st->completed[rows[i]] += num_sched[i];
    }
    *out_total_tokens = static_cast<int32_t>(T);
    return PKV_OK;
}

int pkv_prepare_batch_device(pkv_state *st, const int32_t *d_rows, const int32_t *d_num_sched,
                             int32_t n, int32_t total_tokens, const pkv_batch_out *out,
                             pkv_stream_t stream) {
    if (!st) return PKV_ERR_INVALID_ARG;
    if (n < 0 || n > PKV_MAX_BATCH || total_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!d_rows || !d_num_sched)) return PKV_ERR_INVALID_ARG;
    if (!outputs_ok(st, out, n, total_tokens)) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = pkv::as_stream(stream);
    if (n == 0) {
        PKV_CUDA_TRY(cudaMemsetAsync(out->query_start_loc, 0, sizeof(int32_t), s));
        return PKV_OK;
    }
    pkv::PrepareLaunch in{d_rows, d_num_sched, n, total_tokens};
    return pkv::launch_prepare(st, in, out, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Batch build that allocates nothing: pkv_prepare_batch_static.
//
// The regular host-schedule entry point stages the schedule in device memory
// that pkv_state_create allocated.  This variant takes the request-state
// table as caller-owned device arrays and stages the schedule in a fixed
// array compiled into the library instead, so it needs no device allocation
// at any point.  The array is shared by every call on a device and keeps the
// last call's contents; nothing in it has to start at zero, because each call
// overwrites the [0, n) entries the kernel reads before launching.
// ---------------------------------------------------------------------------
namespace {

// rows at [0, n), counts at the 16-byte aligned offset round_up(n, 4)
static __device__ __align__(256) int32_t g_static_schedule[2 * (PKV_STATIC_MAX_BATCH + 4)];

// Device address of g_static_schedule per device ordinal.  In host code the
// symbol's name is only a host-side stand-in; the address a kernel may use
// comes from cudaGetSymbolAddress with that device current.
int32_t *g_static_schedule_addr[64] = {nullptr};

int static_schedule_address(int device, int32_t **out) {
    if (device < 0 || device >= 64) return PKV_ERR_INVALID_ARG;
    if (!g_static_schedule_addr[device]) {
        void *p = nullptr;
        PKV_CUDA_TRY(cudaGetSymbolAddress(&p, g_static_schedule));
        g_static_schedule_addr[device] = static_cast<int32_t *>(p);
    }
    *out = g_static_schedule_addr[device];
    return PKV_OK;
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
    if (T > INT32_MAX) return PKV_ERR_INVALID_ARG;
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
    int rc = ensure_kernel_attributes(device);
    if (rc != PKV_OK) return rc;
    int32_t *sched = nullptr;
    rc = static_schedule_address(device, &sched);
    if (rc != PKV_OK) return rc;
    const int32_t n4 = (n + 3) & ~3;
    PKV_CUDA_TRY(cudaMemcpyAsync(sched, rows, static_cast<size_t>(n) * 4,
                                 cudaMemcpyHostToDevice, s));
    PKV_CUDA_TRY(cudaMemcpyAsync(sched + n4, num_sched, static_cast<size_t>(n) * 4,
                                 cudaMemcpyHostToDevice, s));
    int num_sms = 0;
    PKV_CUDA_TRY(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device));

    PrepParams p = {};
    p.rows = sched;
    p.counts = sched + n4;
    p.n = n;
    p.T = static_cast<int32_t>(T);
    p.counts_aligned = 1;
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
    int vec = 1;
    for (int g = 0; g < num_groups; g++) {
        if (groups[g].max_blocks_per_req % 4 != 0 ||
            (reinterpret_cast<uintptr_t>(out->block_tables[g]) & 15) ||
            (reinterpret_cast<uintptr_t>(d_block_tables[g]) & 15))
            vec = 0;
    }
    p.vec = vec;
    int64_t alpha = 0;
    p.chunk_off[0] = 0;
    for (int g = 0; g < num_groups; g++) {
        const int32_t w = groups[g].max_blocks_per_req;
        const int32_t units = vec ? w / 4 : w;
        p.chunk_off[g + 1] = p.chunk_off[g] + units;
        p.width[g] = w;
        p.bs[g] = groups[g].block_size;
        int sh = -1;
        if ((groups[g].block_size & (groups[g].block_size - 1)) == 0) {
            sh = 0;
            while ((1 << sh) < groups[g].block_size) sh++;
        }
        p.bs_shift[g] = sh;
        p.num_blocks[g] = groups[g].num_blocks;
        p.table[g] = d_block_tables[g];
        p.out_table[g] = out->block_tables[g];
        p.slots[g] = out->slot_mapping[g];
        alpha += units;
    }
    for (int g = num_groups; g < PKV_MAX_GROUPS; g++) p.chunk_off[g + 1] = p.chunk_off[g];
    p.alpha = alpha;
    p.total_units = alpha * n + T;
    const size_t smem = prepare_smem_bytes(n);
    int per_sm = 0;
    PKV_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prepare_kernel, kThreads,
                                                               smem));
    if (per_sm < 1) per_sm = 1;
    const int64_t max_ctas = static_cast<int64_t>(num_sms) * per_sm;
    int64_t per_cta = (p.total_units + max_ctas - 1) / max_ctas;
    if (per_cta < kMinUnitsPerCta) per_cta = kMinUnitsPerCta;
    p.units_per_cta = per_cta;
    const int64_t grid = (p.total_units + per_cta - 1) / per_cta;
    prepare_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    PKV_CUDA_TRY(cudaGetLastError());
    *out_total_tokens = static_cast<int32_t>(T);
    return PKV_OK;
}
