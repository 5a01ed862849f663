// Paged KV store: copy each new token's K and V line into the cache at its
// slot.  "slot_mapping marks the write slots for this round's new tokens" and
// "each slot storing one token's Key and Value vectors across all attention
// heads" (Multi-Layer Coordinate Conversion Pipeline, page "Deep Dive into
// vLLM's Scheduling Mechanism"); "the slot_id unit is not bytes but a KV
// Cache unit" whose size is heads * head_dim * element size (Address
// Calculation Example).
//
// GB300 design.  A pure HBM-bound byte copy (4 * line_bytes per token: K and V
// each read once and written once).  One warp per token: every lane loads its
// 16-byte vectors of the K and V lines and the slot id (one broadcast load)
// goes out beside them -- the sources do not depend on it -- so one memory
// round trip serves the token and 2 * line_bytes per warp are in flight
// before the stores.
// Sources are read once (ld.global.nc, no L1 allocation) and the cache lines
// are not re-read this step (streaming stores).  When every line start is
// 32-byte aligned each lane moves 32-byte vectors (sm_100+ 256-bit global
// loads/stores), halving the load/store instructions per line.  The grid is a
// whole number of waves over the 152 SMs and grid-strides over tokens; the
// multi-layer variant spreads (layer, token) pairs over the same grid so that
// one launch moves a whole step's worth of layers.
#include "pkv_async.cuh"
#include "pkv_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxLayersPerLaunch = 128;

// One (layer, group) item of a launch: its sources, caches, slot ids and pool.
struct KvLayer {
    const char *k;
    const char *v;
    char *kc;
    char *vc;
    const int64_t *slots;
    int64_t num_slots;
};

// Launch parameters with room for N (layer, group) items.  A launch of a few
// items takes the small block: the parameter block's size is part of every
// launch's latency.
constexpr int kSmallLaunch = 4;
template <int N>
struct KvParamsN {
    KvLayer layer[N];
    int32_t num_layers;
    int32_t T;
    int64_t ks, vs;
    int32_t line;          // bytes, multiple of 16
    int32_t parts_log2;    // each token's lines are moved in 2^parts_log2 equal parts
    int32_t part;          // bytes of K (and of V) per part
    int32_t *err;
};
using KvParams = KvParamsN<kMaxLayersPerLaunch>;

// One lane's piece of a line: 16 or 32 bytes.
template <int B>
struct Vec;
template <>
struct Vec<16> {
    int4 a;
};
template <>
struct Vec<32> {
    int4 a, b;
};

__device__ __forceinline__ void ld_stream(Vec<16> &v, const void *p) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.a.x), "=r"(v.a.y), "=r"(v.a.z), "=r"(v.a.w)
                 : "l"(p));
}
__device__ __forceinline__ void ld_stream(Vec<32> &v, const void *p) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.a.x), "=r"(v.a.y), "=r"(v.a.z), "=r"(v.a.w), "=r"(v.b.x),
                   "=r"(v.b.y), "=r"(v.b.z), "=r"(v.b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st_stream(void *p, const Vec<16> &v) {
    asm volatile("st.global.cs.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.a.x), "r"(v.a.y),
                 "r"(v.a.z), "r"(v.a.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream(void *p, const Vec<32> &v) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "r"(v.a.x), "r"(v.a.y), "r"(v.a.z), "r"(v.a.w), "r"(v.b.x), "r"(v.b.y),
                 "r"(v.b.z), "r"(v.b.w)
                 : "memory");
}

// B = bytes per lane access (16 or 32); kVec = accesses per lane per line when
// the line is a multiple of 32 * B bytes (fully unrolled), 0 = any multiple of B.
template <int B, int kVec, int N>
__global__ void __launch_bounds__(kThreads) kv_write_kernel(const KvParamsN<N> p) {
    pkv::pdl_wait();      // slot_mapping comes from the kernel before
    pkv::pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t per_layer = static_cast<int64_t>(p.T) << p.parts_log2;
    const int64_t items = static_cast<int64_t>(p.num_layers) * per_layer;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); w < items;
         w += stride) {
        const int32_t layer = static_cast<int32_t>(w / per_layer);
        const int64_t r = w - static_cast<int64_t>(layer) * per_layer;
        const int32_t t = static_cast<int32_t>(r >> p.parts_log2);
        const int32_t off = static_cast<int32_t>(r & ((1 << p.parts_log2) - 1)) * p.part;
        const KvLayer L = p.layer[layer];
        const char *ksrc = L.k + t * p.ks + off;
        const char *vsrc = L.v + t * p.vs + off;
        if constexpr (kVec > 0) {
            // the source lines do not depend on the slot: their loads go out
            // beside the slot id's, one memory round trip per item
            Vec<B> a[kVec], b[kVec];
#pragma unroll
            for (int u = 0; u < kVec; u++) {
                ld_stream(a[u], ksrc + (u * 32 + lane) * B);
                ld_stream(b[u], vsrc + (u * 32 + lane) * B);
            }
            const int64_t slot = L.slots[t];
            if (slot < 0) continue;
            if (slot >= L.num_slots) {
                if (lane == 0 && p.err) atomicOr(p.err, PKV_DEVERR_SLOT);
                continue;
            }
            char *kdst = L.kc + slot * p.line + off;
            char *vdst = L.vc + slot * p.line + off;
#pragma unroll
            for (int u = 0; u < kVec; u++) {
                st_stream(kdst + (u * 32 + lane) * B, a[u]);
                st_stream(vdst + (u * 32 + lane) * B, b[u]);
            }
        } else {
            const int64_t slot = L.slots[t];
            if (slot < 0) continue;
            if (slot >= L.num_slots) {
                if (lane == 0 && p.err) atomicOr(p.err, PKV_DEVERR_SLOT);
                continue;
            }
            char *kdst = L.kc + slot * p.line + off;
            char *vdst = L.vc + slot * p.line + off;
            const int chunks = p.part / B;
            for (int c = lane; c < chunks; c += 32) {
                Vec<B> a, b;
                ld_stream(a, ksrc + c * B);
                ld_stream(b, vsrc + c * B);
                st_stream(kdst + c * B, a);
                st_stream(vdst + c * B, b);
            }
        }
    }
}

// Resident CTAs per SM of a kernel variant (cached: the same on every GB300).
int blocks_per_sm(const void *kernel) {
    static const void *keys[16] = {nullptr};
    static int vals[16] = {0};
    for (int i = 0; i < 16; i++) {
        if (keys[i] == kernel) return vals[i];
        if (!keys[i]) {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess ||
                b < 1)
                b = 1;
            keys[i] = kernel;
            vals[i] = b;
            return b;
        }
    }
    return 1;
}

template <int B, int V>
void launch_variant(const KvParams &p, int num_sms, cudaStream_t s) {
    const int64_t items = (static_cast<int64_t>(p.num_layers) * p.T) << p.parts_log2;
    const int64_t need = (items + kWarps - 1) / kWarps;
    if (p.num_layers <= kSmallLaunch) {
        KvParamsN<kSmallLaunch> q;
        for (int l = 0; l < p.num_layers; l++) q.layer[l] = p.layer[l];
        q.num_layers = p.num_layers;
        q.T = p.T;
        q.ks = p.ks;
        q.vs = p.vs;
        q.line = p.line;
        q.parts_log2 = p.parts_log2;
        q.part = p.part;
        q.err = p.err;
        const void *k = reinterpret_cast<const void *>(kv_write_kernel<B, V, kSmallLaunch>);
        // at most one full wave of resident CTAs; they grid-stride over the items
        const int64_t wave = static_cast<int64_t>(num_sms) * blocks_per_sm(k);
        const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
        pkv::launch_pdl(kv_write_kernel<B, V, kSmallLaunch>, dim3(grid), dim3(kThreads), 0, s, q);
        return;
    }
    const void *k = reinterpret_cast<const void *>(kv_write_kernel<B, V, kMaxLayersPerLaunch>);
    const int64_t wave = static_cast<int64_t>(num_sms) * blocks_per_sm(k);
    const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
    pkv::launch_pdl(kv_write_kernel<B, V, kMaxLayersPerLaunch>, dim3(grid), dim3(kThreads), 0, s, p);
}

template <int B>
void launch_width(const KvParams &p, int num_sms, cudaStream_t s) {
    const int per_lane = p.part / (32 * B);
    const bool unrolled = p.part % (32 * B) == 0;
    if (unrolled && per_lane == 1)
        launch_variant<B, 1>(p, num_sms, s);
    else if (unrolled && per_lane == 2)
        launch_variant<B, 2>(p, num_sms, s);
    else if (unrolled && per_lane == 4)
        launch_variant<B, 4>(p, num_sms, s);
    else
        launch_variant<B, 0>(p, num_sms, s);
}

bool aligned_to(const void *q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; }

int launch_kv(KvParams &p, int num_sms, cudaStream_t s) {
    // A launch with few (layer, token) items gives each warp a single
    // load-then-store round, so ramp-up and drain are not amortised: below
    // two items per resident warp (2048 threads an SM), each token's lines
    // are split into two parts moved by different warps, so that a warp's
    // next loads overlap its stores; into four when the items are fewer than
    // a quarter of that (parts stay multiples of 512 bytes).  Measured on the
    // 8192-token single-layer store: two parts 12.6 us, one 12.8 us, four
    // 14.5 us (16-byte accesses); on 38- and 256-token stores four parts are
    // fastest.
    const int64_t base = static_cast<int64_t>(p.num_layers) * p.T;
    const int64_t want = 2 * static_cast<int64_t>(num_sms) * (2048 / 32);
    const int max_log2 = base * 4 <= want ? 2 : 1;
    p.parts_log2 = 0;
    while (p.parts_log2 < max_log2 && (base << p.parts_log2) < want &&
           p.line % ((2 << p.parts_log2) * 512) == 0)
        p.parts_log2++;
    p.part = p.line >> p.parts_log2;
    // 32-byte lane accesses when every line start is 32-byte aligned and a
    // part is whole rounds of 32 x 32 bytes
    bool w32 = p.part % (32 * 32) == 0 && p.ks % 32 == 0 && p.vs % 32 == 0;
    for (int l = 0; l < p.num_layers && w32; l++)
        w32 = aligned_to(p.layer[l].k, 32) && aligned_to(p.layer[l].v, 32) &&
              aligned_to(p.layer[l].kc, 32) && aligned_to(p.layer[l].vc, 32);
    if (w32)
        launch_width<32>(p, num_sms, s);
    else
        launch_width<16>(p, num_sms, s);
    PKV_CUDA_TRY(cudaGetLastError());
    return PKV_OK;
}

int sm_count(int *out) {
    int dev = 0;
    PKV_CUDA_TRY(cudaGetDevice(&dev));
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev]) {
        *out = cached[dev];
        return PKV_OK;
    }
    int n = 0;
    PKV_CUDA_TRY(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
    if (dev >= 0 && dev < 64) cached[dev] = n;
    *out = n;
    return PKV_OK;
}

bool aligned16(const void *p) { return aligned_to(p, 16); }

int check_common(int64_t ks, int64_t vs, int64_t num_slots, int32_t line,
                 const int64_t *slot_mapping, int32_t num_tokens) {
    if (num_tokens < 0 || line <= 0 || num_slots < 0 || ks < 0 || vs < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
    if ((line & 15) || (ks & 15) || (vs & 15)) return PKV_ERR_ALIGN;
    if (num_tokens > 0 && (ks < line || vs < line)) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_kv_cache_write(const void *k, const void *v, int64_t k_stride_bytes,
                       int64_t v_stride_bytes, void *k_cache, void *v_cache, int64_t num_slots,
                       int32_t line_bytes, const int64_t *slot_mapping, int32_t num_tokens,
                       int32_t *d_error, pkv_stream_t stream) {
    int rc = check_common(k_stride_bytes, v_stride_bytes, num_slots, line_bytes, slot_mapping,
                          num_tokens);
    if (rc != PKV_OK) return rc;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_ALIGN;
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != PKV_OK) return rc;
    KvParams p;
    p.layer[0] = KvLayer{static_cast<const char *>(k), static_cast<const char *>(v),
                         static_cast<char *>(k_cache), static_cast<char *>(v_cache),
                         slot_mapping, num_slots};
    p.num_layers = 1;
    p.T = num_tokens;
    p.ks = k_stride_bytes;
    p.vs = v_stride_bytes;
    p.line = line_bytes;
    p.err = d_error;
    return launch_kv(p, sms, pkv::as_stream(stream));
}

int pkv_kv_cache_write_layers(int32_t num_layers, const void *const *k, const void *const *v,
                              int64_t k_stride_bytes, int64_t v_stride_bytes,
                              void *const *k_caches, void *const *v_caches, int64_t num_slots,
                              int32_t line_bytes, const int64_t *slot_mapping,
                              int32_t num_tokens, int32_t *d_error, pkv_stream_t stream) {
    int rc = check_common(k_stride_bytes, v_stride_bytes, num_slots, line_bytes, slot_mapping,
                          num_tokens);
    if (rc != PKV_OK) return rc;
    if (num_layers < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0 || num_layers == 0) return PKV_OK;
    if (!k || !v || !k_caches || !v_caches) return PKV_ERR_INVALID_ARG;
    for (int32_t l = 0; l < num_layers; l++) {
        if (!k[l] || !v[l] || !k_caches[l] || !v_caches[l]) return PKV_ERR_INVALID_ARG;
        if (!aligned16(k[l]) || !aligned16(v[l]) || !aligned16(k_caches[l]) ||
            !aligned16(v_caches[l]))
            return PKV_ERR_ALIGN;
    }
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = pkv::as_stream(stream);
    for (int32_t l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int32_t m = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0
                                                                 : kMaxLayersPerLaunch;
        KvParams p;
        for (int32_t l = 0; l < m; l++)
            p.layer[l] = KvLayer{static_cast<const char *>(k[l0 + l]),
                                 static_cast<const char *>(v[l0 + l]),
                                 static_cast<char *>(k_caches[l0 + l]),
                                 static_cast<char *>(v_caches[l0 + l]), slot_mapping, num_slots};
        p.num_layers = m;
        p.T = num_tokens;
        p.ks = k_stride_bytes;
        p.vs = v_stride_bytes;
        p.line = line_bytes;
        p.err = d_error;
        rc = launch_kv(p, sms, s);
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

int pkv_kv_cache_write_step(int32_t num_items, const pkv_kv_item *items,
                            int64_t k_stride_bytes, int64_t v_stride_bytes, int32_t line_bytes,
                            int32_t num_tokens, int32_t *d_error, pkv_stream_t stream) {
    if (num_items < 0 || (num_items > 0 && !items)) return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < num_items; i++) {
        int rc = check_common(k_stride_bytes, v_stride_bytes, items[i].num_slots, line_bytes,
                              items[i].slot_mapping, num_tokens);
        if (rc != PKV_OK) return rc;
    }
    if (num_items == 0 || num_tokens == 0) {
        return check_common(k_stride_bytes, v_stride_bytes, 0, line_bytes, nullptr, 0);
    }
    for (int32_t i = 0; i < num_items; i++) {
        const pkv_kv_item &it = items[i];
        if (!it.k || !it.v || !it.k_cache || !it.v_cache) return PKV_ERR_INVALID_ARG;
        if (!aligned16(it.k) || !aligned16(it.v) || !aligned16(it.k_cache) ||
            !aligned16(it.v_cache))
            return PKV_ERR_ALIGN;
    }
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = pkv::as_stream(stream);
    for (int32_t i0 = 0; i0 < num_items; i0 += kMaxLayersPerLaunch) {
        const int32_t m = num_items - i0 < kMaxLayersPerLaunch ? num_items - i0
                                                               : kMaxLayersPerLaunch;
        KvParams p;
        for (int32_t i = 0; i < m; i++) {
            const pkv_kv_item &it = items[i0 + i];
            p.layer[i] = KvLayer{static_cast<const char *>(it.k), static_cast<const char *>(it.v),
                                 static_cast<char *>(it.k_cache), static_cast<char *>(it.v_cache),
                                 it.slot_mapping, it.num_slots};
        }
        p.num_layers = m;
        p.T = num_tokens;
        p.ks = k_stride_bytes;
        p.vs = v_stride_bytes;
        p.line = line_bytes;
        p.err = d_error;
        rc = launch_kv(p, sms, s);
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

}  // extern "C"
