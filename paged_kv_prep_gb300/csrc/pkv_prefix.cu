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
// GB300 design.  Digests of all blocks are independent: one thread per block.
// The chain is an affine recurrence, x -> P * x + d, and affine maps compose
// associatively, so a request's keys are a parallel prefix scan over
// (multiplier, addend) pairs -- one CTA per request, tiles of 256 blocks, the
// running composition carried from tile to tile.  The index is an
// open-addressing table of 64-bit keys in device memory (linear probing,
// atomicCAS inserts, bounded probes); a match is one warp per request that
// stops at the first uncached block.
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

// composition of affine maps: first l, then r
struct Affine {
    uint64_t m, a;
};
__device__ __forceinline__ Affine compose(Affine l, Affine r) { return {l.m * r.m, l.a * r.m + r.a}; }

__device__ __forceinline__ Affine shfl_up(Affine v, int d) {
    return {__shfl_up_sync(0xffffffffu, v.m, d), __shfl_up_sync(0xffffffffu, v.a, d)};
}

__global__ void __launch_bounds__(kThreads) block_keys_kernel(
    const int32_t *rows, const int32_t *offsets, int32_t n, const int32_t *tokens,
    int64_t tok_stride, int32_t bs, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    __shared__ Affine s_warp[kWarps];
    __shared__ Affine s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int64_t row = rows[i];
        const int32_t o0 = offsets[i];
        const int32_t nb = offsets[i + 1] - o0;
        const int32_t *tk = tokens + row * tok_stride;
        if (tid == 0) s_carry = {1, 0};
        __syncthreads();
        for (int32_t base = 0; base < nb; base += kThreads) {
            const int32_t j = base + tid;
            Affine v = {1, 0};
            if (j < nb) {
                uint64_t h = kBasis;
                const int32_t *b = tk + static_cast<int64_t>(j) * bs;
                for (int32_t k = 0; k < bs; k++) {
                    const uint32_t t = static_cast<uint32_t>(b[k]);
#pragma unroll
                    for (int x = 0; x < 4; x++) {
                        h ^= (t >> (8 * x)) & 0xffu;
                        h *= kPrime;
                    }
                }
                v = {kPrime, h};
            }
            // inclusive scan of the tile's maps
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const Affine o = shfl_up(v, d);
                if (lane >= d) v = compose(o, v);
            }
            if (lane == 31) s_warp[warp] = v;
            __syncthreads();
            Affine before = s_carry;
            for (int w = 0; w < warp; w++) before = compose(before, s_warp[w]);
            const Affine full = compose(before, v);
            if (j < nb) keys[o0 + j] = full.m * kBasis + full.a;
            __syncthreads();
            if (tid == kThreads - 1) s_carry = full;   // the tile's last composition
            __syncthreads();
        }
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

__global__ void __launch_bounds__(kThreads) match_kernel(
    const unsigned long long *table_keys, const int32_t *table_ids, int64_t mask,
    const uint64_t *keys, const int32_t *offsets, const int32_t *max_hits, int32_t n,
    int32_t *hit_blocks, int32_t *hit_ids) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); w < n;
         w += stride) {
        const int32_t o0 = offsets[w];
        const int32_t nk = offsets[w + 1] - o0;
        const int32_t cap = min(nk, max(0, max_hits[w]));
        int32_t hits = 0;
        bool open = true;
        for (int32_t base = 0; base < nk; base += 32) {
            const int32_t j = base + lane;
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
            // hits continue while every earlier block of the request hit
            const unsigned miss = __ballot_sync(0xffffffffu, !found);
            const int first_miss = miss ? __ffs(miss) - 1 : 32;
            if (open) {
                if (j < nk) hit_ids[o0 + j] = lane < first_miss ? id : -1;
                if (first_miss < 32) {
                    hits = base + first_miss;
                    open = false;
                }
            } else if (j < nk) {
                hit_ids[o0 + j] = -1;
            }
        }
        if (open) hits = nk;
        if (lane == 0) hit_blocks[w] = min(hits, cap);
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
    // one host-to-device copy: rows, then offsets at a 16-byte aligned offset
    const int32_t n4 = (n + 3) & ~3;
    int status;
    char *buf = st->ring.reserve(static_cast<size_t>(n4 + n + 1) * 4, &status);
    if (!buf) return status;
    memcpy(buf, rows, static_cast<size_t>(n) * 4);
    memcpy(buf + static_cast<size_t>(n4) * 4, out_offsets, static_cast<size_t>(n + 1) * 4);
    cudaStream_t s = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(st->d_sched, buf, static_cast<size_t>(n4 + n + 1) * 4,
                                    cudaMemcpyHostToDevice, s);
    const int rc = st->ring.fence(s);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return PKV_ERR_CUDA;
    }
    if (rc != PKV_OK) return rc;
    const unsigned grid = static_cast<unsigned>(n < st->num_sms * 8 ? n : st->num_sms * 8);
    PKV_CUDA_TRY(launch_pdl(block_keys_kernel, dim3(grid), dim3(kThreads), 0, s,
                            static_cast<const int32_t *>(st->d_sched),
                            static_cast<const int32_t *>(st->d_sched + n4), n,
                            static_cast<const int32_t *>(st->d_tokens),
                            static_cast<int64_t>(st->max_len), block_size, d_keys));
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
    PKV_CUDA_TRY(launch_pdl(match_kernel, dim3(grid_for(n, kWarps, sms)), dim3(kThreads), 0,
                            as_stream(stream), pc->d_keys, pc->d_ids, pc->capacity - 1, d_keys,
                            d_offsets, d_max_hits, n, d_hit_blocks, d_hit_ids));
    return PKV_OK;
}

}  // extern "C"
