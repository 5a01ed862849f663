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
// first pass spreads every block of every request evenly over the grid, one
// thread per block reading its tokens from shared memory, where the tile was
// staged with coalesced loads.  The chain is an affine recurrence,
// x -> P * x + d, and affine maps compose associatively, so the second pass
// turns each request's digests into keys with a parallel prefix scan over
// (multiplier, addend) pairs -- one CTA per request, 256 blocks per round.  The index is an
// open-addressing table of 64-bit keys in device memory (linear probing,
// atomicCAS inserts, bounded probes); a match is one CTA per request probing
// 256 keys per round and stopping at the first uncached block.
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
constexpr size_t kMaxKeysSmem = 224 * 1024;   // staged tokens of one tile of blocks

// composition of affine maps: first l, then r
struct Affine {
    uint64_t m, a;
};
__device__ __forceinline__ Affine compose(Affine l, Affine r) { return {l.m * r.m, l.a * r.m + r.a}; }

__device__ __forceinline__ Affine shfl_up(Affine v, int d) {
    return {__shfl_up_sync(0xffffffffu, v.m, d), __shfl_up_sync(0xffffffffu, v.a, d)};
}

// Shared-memory row pitch of one block's tokens: odd, so thread t reading
// word t * pitch + k hits bank (t + k) mod 32 -- no conflicts.
__host__ __device__ inline int32_t token_pitch(int32_t bs) { return (bs & 1) ? bs : bs + 1; }

// Pass 1: the FNV-1a digest of every block of every request, flat over all
// blocks in tiles of 256 (every CTA gets the same work, whatever the mix of
// request lengths).  Each thread finds its block's request in the staged
// offsets, the tile's tokens are staged into shared memory with coalesced
// loads (one odd-pitch row per block), and each thread digests its row.
// The digests go to keys[], where pass 2 turns them into chained keys.
__global__ void __launch_bounds__(kThreads) block_digest_kernel(
    const int32_t *rows, const int32_t *offsets, int32_t n, const int32_t *tokens,
    int64_t tok_stride, int32_t bs, int32_t total, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t smem[];
    const int32_t pitch = token_pitch(bs);
    int32_t *s_tok = smem;                      // [kThreads][pitch]
    int32_t *s_off = smem + kThreads * pitch;   // [n + 1]
    __shared__ const int32_t *s_src[kThreads];
    const int tid = threadIdx.x;
    for (int32_t e = tid; e <= n; e += kThreads) s_off[e] = offsets[e];
    __syncthreads();
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads; base < total;
         base += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int32_t j = static_cast<int32_t>(base) + tid;
        if (j < total) {
            // the request whose blocks contain j: last i with s_off[i] <= j
            int lo = 0, hi = n;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= j) lo = mid; else hi = mid;
            }
            s_src[tid] = tokens + static_cast<int64_t>(rows[lo]) * tok_stride +
                         static_cast<int64_t>(j - s_off[lo]) * bs;
        }
        __syncthreads();
        const int32_t tile_blocks = static_cast<int32_t>(total - base < kThreads ? total - base : kThreads);
        const int32_t tile_tokens = tile_blocks * bs;
        {
            const int32_t step_blk = kThreads / bs, step_off = kThreads % bs;
            int32_t blk = tid / bs, off = tid - (tid / bs) * bs;
            for (int32_t e0 = 0; e0 < tile_tokens; e0 += 8 * kThreads) {
                int32_t val[8], dst[8];
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int32_t e = e0 + u * kThreads + tid;
                    dst[u] = e < tile_tokens ? blk * pitch + off : -1;
                    val[u] = e < tile_tokens ? s_src[blk][off] : 0;
                    blk += step_blk;
                    off += step_off;
                    if (off >= bs) {
                        off -= bs;
                        blk++;
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; u++)
                    if (dst[u] >= 0) s_tok[dst[u]] = val[u];
            }
        }
        __syncthreads();
        if (j < total) {
            uint64_t h = kBasis;
            const int32_t *row = s_tok + tid * pitch;
            for (int32_t k = 0; k < bs; k++) {
                const uint32_t t = static_cast<uint32_t>(row[k]);
#pragma unroll
                for (int x = 0; x < 4; x++) {
                    h ^= (t >> (8 * x)) & 0xffu;
                    h *= kPrime;
                }
            }
            keys[j] = h;
        }
        __syncthreads();
    }
}

// Pass 2: each request's chain, key_j = key_{j-1} * P + digest_j, as a
// block-wide scan of affine maps (one CTA per request, 256 blocks per round,
// the running composition carried from round to round), in place.
__global__ void __launch_bounds__(kThreads) block_chain_kernel(const int32_t *offsets,
                                                               int32_t n, uint64_t *keys) {
    pdl_wait();
    pdl_trigger();
    __shared__ Affine s_warp[kWarps];
    __shared__ Affine s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t o0 = offsets[i];
        const int32_t nb = offsets[i + 1] - o0;
        if (tid == 0) s_carry = {1, 0};
        __syncthreads();
        for (int32_t base = 0; base < nb; base += kThreads) {
            const int32_t j = base + tid;
            Affine v = {1, 0};
            if (j < nb) v = {kPrime, keys[o0 + j]};
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
            if (tid == kThreads - 1) s_carry = full;   // the round's last composition
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
    const size_t smem = (static_cast<size_t>(kThreads) * token_pitch(block_size) + n + 1) * 4;
    if (smem > kMaxKeysSmem) return PKV_ERR_INVALID_ARG;   // block_size above ~150 tokens
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
    const int64_t tiles = (total + kThreads - 1) / kThreads;
    const int64_t wave = static_cast<int64_t>(st->num_sms) * per_sm;
    const unsigned grid1 = static_cast<unsigned>(tiles < wave ? tiles : wave);
    const int32_t *d_rows = st->d_sched;
    const int32_t *d_off = st->d_sched + n4;
    PKV_CUDA_TRY(launch_pdl(block_digest_kernel, dim3(grid1), dim3(kThreads), smem, s, d_rows,
                            d_off, n, static_cast<const int32_t *>(st->d_tokens),
                            static_cast<int64_t>(st->max_len), block_size,
                            static_cast<int32_t>(total), d_keys));
    const int64_t wave2 = static_cast<int64_t>(st->num_sms) * (2048 / kThreads);
    const unsigned grid2 = static_cast<unsigned>(n < wave2 ? n : wave2);
    PKV_CUDA_TRY(launch_pdl(block_chain_kernel, dim3(grid2), dim3(kThreads), 0, s, d_off, n,
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
    PKV_CUDA_TRY(launch_pdl(match_kernel, dim3(grid_for(n, 1, sms)), dim3(kThreads), 0,
                            as_stream(stream), pc->d_keys, pc->d_ids, pc->capacity - 1, d_keys,
                            d_offsets, d_max_hits, n, d_hit_blocks, d_hit_ids));
    return PKV_OK;
}

}  // extern "C"
