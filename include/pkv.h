/*
 * pkv.h -- C ABI of paged_kv_prep_gb300: per-step input preparation and
 * paged-KV store for a vLLM-style worker, on one GB300 (sm_103a).
 *
 * The operations follow the pages "Deep Dive into vLLM's Scheduling Mechanism:
 * The Complete CPU-to-GPU Mapping Pipeline" (kongchang.com, English; Chinese
 * original "vLLM调度机制深度解析") and "从源码读 vLLM Scheduler"
 * (caffein.top), cited below by page and section.
 *
 * Conventions
 *   - Every call returns a pkv_status (0 = PKV_OK, negative = error).  No call
 *     aborts, prints or traps.
 *   - "device" pointers are CUDA global-memory pointers on the state's device;
 *     "host" pointers are ordinary CPU memory and may be released as soon as
 *     the call returns (the library copies them into its own pinned ring).
 *   - Streams are cudaStream_t values passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work on the stream and return; only the calls
 *     marked "synchronous" wait for the GPU.  A pinned-ring wrap may wait for
 *     earlier copies from the same ring to finish (back-pressure).
 *   - One pkv_state belongs to one stream at a time; the library is not
 *     thread-safe for a given state.
 *   - All integer arrays are int32 except slot ids, which are int64 so that
 *     slot * line_bytes never overflows for the caller.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_MAX_GROUPS 8       /* KV-cache groups per state */
#define PKV_MAX_BATCH 16384    /* requests per prepare call */
#define PKV_STATIC_MAX_BATCH 4096  /* requests per pkv_prepare_batch_static call */
#define PKV_MAX_TOKENS (1 << 26)   /* scheduled tokens per prepare call: T < 2^26 */

typedef void *pkv_stream_t;    /* a cudaStream_t */

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,  /* a pointer, size or value is out of range */
    PKV_ERR_FULL = -2,         /* no free request row */
    PKV_ERR_NOT_ACTIVE = -3,   /* the row holds no live request */
    PKV_ERR_CAPACITY = -4,     /* a position, token id or block is missing */
    PKV_ERR_ALIGN = -5,        /* a pointer, stride or size is not 16-B aligned */
    PKV_ERR_CUDA = -6,         /* a CUDA call failed; see pkv_last_cuda_error */
    PKV_ERR_DEVICE = -7        /* the device error word was set (pkv_get_error) */
} pkv_status;

/* Bits of the device error word (pkv_get_error).  A kernel that meets a bad
   input sets a bit, skips that element (writing -1 where an output element
   stands for it) and carries on; it never traps. */
enum {
    PKV_DEVERR_ROW = 1,        /* a scheduled row is outside the table */
    PKV_DEVERR_COUNT = 2,      /* a scheduled count < 1, or counts do not sum to T */
    PKV_DEVERR_POSITION = 4,   /* a position is at or past max_model_len */
    PKV_DEVERR_BLOCK = 8,      /* a position's block is missing (-1 / past W) */
    PKV_DEVERR_SLOT = 16,      /* a KV-store slot is at or past num_slots */
    PKV_DEVERR_TIMEOUT = 32,   /* a bounded wait inside a kernel gave up */
    PKV_DEVERR_TABLE_FULL = 64, /* a prefix-cache insert found no free slot */
    PKV_DEVERR_OUTPUT_FULL = 128, /* an output array was too small for the entries */
    PKV_DEVERR_DUP = 256       /* a device schedule lists a row twice (all but one listing get -1) */
};

/* prepare flags */
#define PKV_ADVANCE 1          /* after preparing, completed_tokens += scheduled */
#define PKV_LIVE_TABLES 2      /* gather only the live block-table entries (see below) */
#define PKV_SCHEDULE_SETTLED 4 /* device schedule only: its arrays were not written by the
                                  kernel launched just before on the stream, so the batch
                                  build may check and rank them while that kernel finishes */

/* One KV-cache group: "Different KV Cache groups generate their own
   block_tables and slot_mappings" (Address Calculation Example).  block_size
   is tokens per physical block; max_blocks_per_req is the block-table width W;
   num_blocks is the size of the group's physical pool (ids 0..num_blocks-1;
   -1 is the null id). */
typedef struct {
    int32_t block_size;
    int32_t max_blocks_per_req;
    int64_t num_blocks;
} pkv_group_spec;

typedef struct pkv_state pkv_state;   /* opaque */

/*
 * Create the worker's persistent request-state table on the current CUDA
 * device ("request_state" and "block_table", Worker Request State
 * Management).  It holds, per row: completed_tokens, the known token ids
 * (max_model_len int32 each) and, per group, a block-table row of W int32
 * (all -1 when empty).  max_reqs rows (1..65536); 1 <= num_groups <=
 * PKV_MAX_GROUPS; groups[] is host memory.  The state owns its device memory
 * and a pinned host ring of ring_bytes (0 = 64 MiB) used to stage host
 * inputs.  Rows are handed out lowest-first and recycled on removal
 * ("Design Logic Behind the Dual-Index System").  The tables are initialised
 * on stream s.
 */
int pkv_state_create(pkv_state **out, int32_t max_reqs, int32_t max_model_len,
                     int32_t num_groups, const pkv_group_spec *groups,
                     int64_t ring_bytes, pkv_stream_t s);

/* Synchronous: waits for the state's outstanding work, frees everything. */
int pkv_state_destroy(pkv_state *st);

/*
 * add_request(): "initializes state and block_table for a new request"
 * (Worker Request State Management).  Takes the lowest free row, stores
 * n_tokens known token ids (host token_ids[n_tokens]; prompt plus any sampled
 * tokens), sets completed_tokens = num_computed_tokens (0 for a fresh request;
 * more for a prefix-cache hit or a resumed request), and fills each group's
 * block-table row with block_ids[g][0..n_blocks[g]) followed by -1.
 * block_ids is a host array of num_groups host pointers; n_blocks is host
 * int32[num_groups].  Block ids must be -1 or < num_blocks; -1 entries may
 * only form a prefix (blocks freed out of a sliding window, "allocate_slots()"
 * on the page "从源码读 vLLM Scheduler").  Returns the row in *out_row.
 * Errors: PKV_ERR_FULL (no free row), PKV_ERR_INVALID_ARG.
 */
int pkv_add_request(pkv_state *st, const int32_t *token_ids, int32_t n_tokens,
                    int32_t num_computed_tokens, const int32_t *const *block_ids,
                    const int32_t *n_blocks, int32_t *out_row, pkv_stream_t s);

/*
 * update_request(): "appends newly allocated block IDs for an already
 * registered request" (Worker Request State Management).  Appends
 * new_block_ids[g][0..n_new_blocks[g]) after the row's current blocks, appends
 * n_new_tokens token ids (e.g. the token sampled last step), and, when
 * num_computed_tokens >= 0, sets completed_tokens to it (the count the
 * scheduler reports for a cached request, "SchedulerOutput" section of
 * "从源码读 vLLM Scheduler"); -1 keeps it.  new_block_ids / n_new_blocks may
 * be NULL for no new blocks.  Errors: PKV_ERR_NOT_ACTIVE, PKV_ERR_CAPACITY
 * (table row or token row would overflow), PKV_ERR_INVALID_ARG.
 */
int pkv_update_request(pkv_state *st, int32_t row, const int32_t *const *new_block_ids,
                       const int32_t *n_new_blocks, const int32_t *new_token_ids,
                       int32_t n_new_tokens, int32_t num_computed_tokens, pkv_stream_t s);

/*
 * A finished request returns its row for reuse ("when a request completes,
 * the index is recycled for reuse", Design Logic Behind the Dual-Index
 * System; finished_req_ids in "SchedulerOutput").  The row is reset:
 * completed_tokens = 0, block-table rows all -1.  Errors: PKV_ERR_NOT_ACTIVE,
 * PKV_ERR_INVALID_ARG.
 */
int pkv_remove_request(pkv_state *st, int32_t row, pkv_stream_t s);

/*
 * One step's scheduler output, as the worker applies it to its persistent
 * state ("SchedulerOutput" section of "从源码读 vLLM Scheduler": requests the
 * worker sees for the first time carry full information, requests it already
 * knows carry only what changed, and finished requests are cleaned up).  All
 * arrays are host memory; ragged lists are CSR: offsets[k]..offsets[k+1].
 */
typedef struct {
    /* finished requests: their rows are freed and reset */
    int32_t num_finished;
    const int32_t *finished_rows;                     /* [num_finished] */
    /* new requests: each takes the lowest free row (after the frees) */
    int32_t num_new;
    const int32_t *new_token_offsets;                 /* [num_new + 1] */
    const int32_t *new_token_ids;
    const int32_t *new_num_computed;                  /* [num_new] */
    const int32_t *new_block_offsets[PKV_MAX_GROUPS]; /* per group [num_new + 1] */
    const int32_t *new_block_ids[PKV_MAX_GROUPS];
    /* cached requests: appended token ids and block ids, computed count */
    int32_t num_cached;
    const int32_t *cached_rows;                       /* [num_cached], distinct */
    const int32_t *cached_token_offsets;              /* [num_cached + 1] */
    const int32_t *cached_token_ids;
    const int32_t *cached_num_computed;               /* [num_cached], -1 keeps */
    const int32_t *cached_block_offsets[PKV_MAX_GROUPS];
    const int32_t *cached_block_ids[PKV_MAX_GROUPS];
} pkv_step_delta;

/*
 * Apply one step's scheduler output to the state in the order the runner
 * uses: free the finished rows, add the new requests, then update the cached
 * ones -- the same result as pkv_remove_request, pkv_add_request and
 * pkv_update_request called one by one in that order, but validated as a
 * whole (nothing changes if any part is invalid) and written by one kernel
 * from one host-to-device copy (more only if the packed delta exceeds a
 * quarter of the pinned ring).  out_new_rows (host [num_new]) receives the
 * rows given to the new requests.  Per-group pointers may be NULL when no
 * request of that kind has blocks in that group.  Errors: those of the
 * individual calls, plus PKV_ERR_INVALID_ARG for a row listed twice.
 */
int pkv_apply_step(pkv_state *st, const pkv_step_delta *delta, int32_t *out_new_rows,
                   pkv_stream_t s);

/* Caller-owned device output buffers of one prepare call (n requests, T
   tokens; num_groups entries of the per-group arrays are used). */
typedef struct {
    int32_t *index_mapping;     /* [n]    batch_index -> request_state_index */
    int32_t *query_start_loc;   /* [n+1]  prefix sum of scheduled counts */
    int32_t *seq_lens;          /* [n]    completed + scheduled */
    int32_t *positions;         /* [T]    position of each flat token */
    int32_t *input_ids;         /* [T]    token id at that position */
    int32_t *block_tables[PKV_MAX_GROUPS];  /* [n][W_g] gathered table rows */
    int64_t *slot_mapping[PKV_MAX_GROUPS];  /* [T] write slot per token */
} pkv_batch_out;

/*
 * Build one step's batch from the schedule output (one fused kernel).
 *   rows[n], num_sched[n]: host arrays, the scheduled requests' rows and
 *   num_scheduled_tokens, in schedule-output order.
 * Steps (all on the GPU):
 *   - sort the requests by num_sched, ascending, equal counts in schedule
 *     order, into batch order; index_mapping[b] = row of batch entry b
 *     ("Extracting the Execution Batch from Global State");
 *   - query_start_loc[0] = 0, query_start_loc[b+1] = query_start_loc[b] +
 *     n_b; positions[t] = completed + (t - query_start_loc[b]); input_ids[t] =
 *     token id at that position ("Contiguous Token Sequence Processing");
 *     seq_lens[b] = completed + n_b ("Complete Input Preparation for the
 *     Attention Module");
 *   - per group g: slot_mapping[g][t] = block_table[row][pos / bs] * bs +
 *     pos % bs and block_tables[g][b][0..W_g) = the row's block-table row
 *     ("Multi-Layer Coordinate Conversion Pipeline", "Address Calculation
 *     Example").
 * flags: PKV_ADVANCE adds n_b to each request's completed_tokens afterwards.
 * PKV_LIVE_TABLES writes, of each gathered block-table row, only the entries
 * attention can read -- j < ceil(seq_lens[b] / block_size_g), the blocks of
 * the request's history and this step ("Complete Input Preparation for the
 * Attention Module": seq_lens tells the kernel the KV range to attend to);
 * the rest of the row is left unspecified (whole 4/16/32-byte chunks are
 * copied, so a few entries past the live ones may be written too).
 * The host checks, before launching, that every row is live and listed once,
 * n_b >= 1, completed + n_b <= known tokens, and every scheduled position has
 * a block in every group.  *out_total_tokens receives T = sum n_b.  n = 0 is
 * allowed (query_start_loc[0] = 0 is written).  Output pointers must be
 * device memory sized as above; block_tables[g] rows are copied with 16-byte
 * vectors when every row start is 16-byte aligned.  rows and num_sched may
 * be released when the call returns: up to 256 requests (without
 * PKV_ADVANCE) they are copied into the kernel's launch parameters, larger
 * schedules into the state's pinned staging ring and from there to the GPU.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_NOT_ACTIVE, PKV_ERR_CAPACITY,
 * PKV_ERR_CUDA.
 */
int pkv_prepare_batch(pkv_state *st, const int32_t *rows, const int32_t *num_sched,
                      int32_t n, int32_t flags, const pkv_batch_out *out,
                      int32_t *out_total_tokens, pkv_stream_t s);

/*
 * The same batch build with the schedule already in device memory
 * (d_rows[n], d_num_sched[n]) and its token total T given by the caller, for
 * callers that keep the schedule on the GPU or capture the step in a CUDA
 * graph.  No host validation: the kernel checks rows, counts (each >= 1,
 * summing to T), positions and blocks, sets the device error word on a
 * violation and writes -1 for the affected outputs.  A row listed more than
 * once ("Extracting the Execution Batch from Global State": one batch row
 * per request) is kept by one listing -- whichever claims it first on the
 * GPU, so not always the first in schedule order -- and every other listing
 * is ranked as usual but gets -1 for all its outputs (no two tokens share a
 * slot), with PKV_DEVERR_DUP set.  The claims use a per-row stamp in the
 * state (8 bytes per row) tagged with a call number.  flags: PKV_LIVE_TABLES
 * as for pkv_prepare_batch; PKV_SCHEDULE_SETTLED when d_rows / d_num_sched
 * were not written by the kernel launched just before on s (the kernel may
 * then check and rank them while that kernel finishes; without the flag it
 * waits first); PKV_ADVANCE is not accepted here (the host keeps no record
 * of device-side schedules).
 */
int pkv_prepare_batch_device(pkv_state *st, const int32_t *d_rows,
                             const int32_t *d_num_sched, int32_t n, int32_t total_tokens,
                             int32_t flags, const pkv_batch_out *out, pkv_stream_t s);

/*
 * The batch build of pkv_prepare_batch for callers that cannot allocate
 * device memory.  (No counterpart on the pages: this is a deployment
 * variant, not a step of the method.)
 *
 * Who needs it: a serving engine that hands nearly all free HBM to its paged
 * KV cache at start-up and forbids later allocations, so that a library
 * allocating at run time would fail or fragment the pool; plugin and
 * callback interfaces of other runtimes, which must not allocate while they
 * run; and code that has no pkv_state, because creating one allocates the
 * request-state table and the schedule staging buffer.  This entry point
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The caller owns the request-state table and passes it as device arrays in
 * the layout pkv_state keeps: d_completed[max_reqs], d_token_ids
 * [max_reqs][max_model_len], and per group d_block_tables[g]
 * [max_reqs][groups[g].max_blocks_per_req] (-1 = no block).  rows[n] and
 * num_sched[n] are host arrays in schedule-output order; out is as for
 * pkv_prepare_batch; d_error is an optional device int32 that receives the
 * PKV_DEVERR_* bits of the kernel's checks (as pkv_prepare_batch_device
 * does: bad positions or missing blocks give -1 outputs).  The host checks
 * that rows lie in [0, max_reqs), are distinct, and that counts are >= 1.
 *
 * Where the schedule goes: up to 256 requests travel in the kernel's
 * parameter block (no copy, no shared state).  A larger schedule is staged
 * in one fixed array compiled into the library: 2 * (PKV_STATIC_MAX_BATCH +
 * 4) int32 (32 KiB), held by every GPU that loads the library until the
 * process exits.  n > PKV_STATIC_MAX_BATCH is rejected with
 * PKV_ERR_INVALID_ARG.  All calls on a device share that array: calls with
 * more than 256 requests whose work overlaps on the GPU (different streams
 * without ordering between them) race on it and must not be issued; calls
 * from several host threads at once are not supported.  It keeps the last
 * call's contents; every call overwrites what its kernel reads.  The host
 * arrays are copied (through a fixed host buffer, as pageable memory) before
 * the call returns, so rows and num_sched -- pinned or not -- may be reused
 * or released as soon as it returns.  A call with more than 256 requests
 * looks up the array's device address (cudaGetSymbolAddress, with the
 * calling thread's current device) and is refused with PKV_ERR_INVALID_ARG
 * while s is being captured into a CUDA graph (a recorded copy would read
 * the host buffer again at replay).
 *
 * Errors: PKV_ERR_INVALID_ARG for null pointers, sizes out of range, a row
 * outside [0, max_reqs), a count < 1, a row listed twice, or T >=
 * PKV_MAX_TOKENS; PKV_ERR_CUDA.
 */
int pkv_prepare_batch_static(const int32_t *d_completed, const int32_t *d_token_ids,
                             int32_t max_reqs, int32_t max_model_len, int32_t num_groups,
                             const pkv_group_spec *groups,
                             const int32_t *const *d_block_tables, const int32_t *rows,
                             const int32_t *num_sched, int32_t n, const pkv_batch_out *out,
                             int32_t *d_error, int32_t *out_total_tokens, pkv_stream_t s);

/*
 * Paged (CSR) block table of a prepared batch, for attention kernels that
 * take a page list instead of padded table rows.  "Complete Input
 * Preparation for the Attention Module": the block tables and seq_lens
 * together tell attention which physical blocks hold each request's KV and
 * how far its history reaches, so request b reads the first
 * pages_b = ceil(seq_lens[b] / bs) entries of its row in group `group`.  This
 * call lists exactly those entries, request after request in batch order:
 *   d_kv_indptr[n+1]   kv_indptr[0] = 0, kv_indptr[b+1] = kv_indptr[b] +
 *                      pages_b (the CSR encoding that query_start_loc uses,
 *                      "Contiguous Token Sequence Processing");
 *   d_kv_indices[capacity]  entry kv_indptr[b] + j = block_table[row_b][j],
 *                      j < pages_b, copied verbatim (a block freed out of a
 *                      sliding window is listed as -1);
 *   d_last_page_len[n] (may be NULL) seq_lens[b] - (pages_b - 1) * bs, the
 *                      positions held by the request's last listed block.
 * d_index_mapping[n] and d_seq_lens[n] are a prepared batch's outputs (any
 * call of the pkv_prepare_batch family, issued before this one on the same
 * stream).  All arrays are device memory owned by the caller.
 * Device checks, reported in the state's error word (pkv_get_error): a row
 * outside the table (PKV_DEVERR_ROW), seq_lens[b] < 1 (PKV_DEVERR_COUNT) or
 * more than W_g pages (PKV_DEVERR_BLOCK) give that request 0 pages and
 * last_page_len 0; more than `capacity` entries in all set
 * PKV_DEVERR_OUTPUT_FULL, and entries at or past capacity are not written
 * (kv_indptr still counts them).  capacity = n * W_g always suffices.
 * Host checks (PKV_ERR_INVALID_ARG): the group, 0 <= n <= PKV_MAX_BATCH,
 * non-null arrays, n * W_g < 2^31.  One kernel: every CTA turns the page
 * counts into offsets in shared memory, then the entries are split evenly
 * over the grid.  n = 0 writes kv_indptr[0] = 0.
 */
int pkv_kv_indices(pkv_state *st, int32_t group, const int32_t *d_index_mapping,
                   const int32_t *d_seq_lens, int32_t n, int32_t *d_kv_indptr,
                   int32_t *d_kv_indices, int64_t capacity, int32_t *d_last_page_len,
                   pkv_stream_t s);

/*
 * Store each new token's K and V vectors at its slot: "slot_mapping ...
 * specifying which physical locations the newly computed KV vectors should be
 * stored in", a slot holding "one token's Key and Value vectors across all
 * attention heads" (Multi-Layer Coordinate Conversion Pipeline).  One call per
 * group per layer.
 *   k, v:        device, token t's line at k + t * k_stride_bytes
 *                (line_bytes = heads * head_dim * element size), e.g. [T][H][D];
 *   k_cache, v_cache: device, num_slots lines of line_bytes each
 *                ([num_blocks * block_size][H][D]); slot s starts at
 *                s * line_bytes;
 *   slot_mapping: device int64[num_tokens]; negative slots are skipped;
 *   d_error:     optional device int32 error word (e.g. pkv_state_error_word);
 *                a slot >= num_slots sets PKV_DEVERR_SLOT there and is skipped.
 * A pure byte copy: fp8/bf16/fp16 bits arrive unchanged.  k, v, the caches,
 * both strides and line_bytes must be multiples of 16 bytes (PKV_ERR_ALIGN).
 */
int pkv_kv_cache_write(const void *k, const void *v, int64_t k_stride_bytes,
                       int64_t v_stride_bytes, void *k_cache, void *v_cache,
                       int64_t num_slots, int32_t line_bytes, const int64_t *slot_mapping,
                       int32_t num_tokens, int32_t *d_error, pkv_stream_t s);

/*
 * The KV store for num_layers layers that share one slot_mapping (all layers
 * of one KV-cache group in a step), in one launch.  k, v, k_caches, v_caches
 * are host arrays of num_layers device pointers; every layer uses the same
 * strides, line_bytes and num_slots.  Same rules as pkv_kv_cache_write.
 */
int pkv_kv_cache_write_layers(int32_t num_layers, const void *const *k,
                              const void *const *v, int64_t k_stride_bytes,
                              int64_t v_stride_bytes, void *const *k_caches,
                              void *const *v_caches, int64_t num_slots,
                              int32_t line_bytes, const int64_t *slot_mapping,
                              int32_t num_tokens, int32_t *d_error, pkv_stream_t s);

/* One (layer, group) item of a step's KV store: its K/V sources, its caches,
   its group's slot_mapping and the size of its group's pool in slots. */
typedef struct {
    const void *k;
    const void *v;
    void *k_cache;
    void *v_cache;
    const int64_t *slot_mapping;
    int64_t num_slots;
} pkv_kv_item;

/*
 * The whole step's KV store in one launch: every (layer, group) item of the
 * step, each with its own slot_mapping and pool ("Different KV Cache groups
 * generate their own block_tables and slot_mappings", Address Calculation
 * Example).  items is a host array of num_items; all items share the source
 * strides, line_bytes and num_tokens (one step's tokens).  Same rules as
 * pkv_kv_cache_write for each item.
 */
int pkv_kv_cache_write_step(int32_t num_items, const pkv_kv_item *items,
                            int64_t k_stride_bytes, int64_t v_stride_bytes, int32_t line_bytes,
                            int32_t num_tokens, int32_t *d_error, pkv_stream_t s);

/* ------------------------------------------------------------------------ */
/* Prefix cache ("Prefix Cache" section of "从源码读 vLLM Scheduler": the    */
/* hash covers a token block and its prefix context; a hit reuses the        */
/* block's K/V; hits are limited to num_tokens - 1).  The page does not fix  */
/* the hash; this library's keys are:                                        */
/*   digest_j = FNV-1a 64 over the 4*bs little-endian bytes of block j's ids */
/*   key_j    = key_{j-1} * 0x100000001b3 + digest_j (mod 2^64),             */
/*              key_{-1} = 0xcbf29ce484222325                                */
/* ------------------------------------------------------------------------ */

/*
 * Keys of the full blocks (block_size tokens each) of the known token ids of
 * rows[0..n) (host array of live rows).  out_offsets (host [n+1]) receives
 * the CSR offsets: row i's keys are d_keys[out_offsets[i] .. out_offsets[i+1]),
 * floor(known tokens / block_size) of them.  With d_keys NULL only the
 * offsets are computed (a size query).  d_keys is device memory of capacity
 * entries (PKV_ERR_CAPACITY if too small).  Any block_size >= 1.  The
 * block digests spread evenly over the GPU's threads (one block each, read
 * as 16-byte vectors when block_size and the row length are multiples of 4
 * tokens, else staged by warps), then each request's digests are chained: a
 * warp per request of up to 256 blocks, a CTA per longer one.
 */
int pkv_block_keys(pkv_state *st, const int32_t *rows, int32_t n, int32_t block_size,
                   int32_t *out_offsets, uint64_t *d_keys, int64_t capacity, pkv_stream_t s);

typedef struct pkv_prefix_cache pkv_prefix_cache;   /* device index: key -> block id */

/* An empty index of `capacity` slots (a power of two, >= 2) on the current
   device.  Key 0 is reserved for empty slots: a block whose key is 0 is never
   cached. */
int pkv_prefix_cache_create(pkv_prefix_cache **out, int64_t capacity, pkv_stream_t s);

/* Synchronous: frees the index. */
int pkv_prefix_cache_destroy(pkv_prefix_cache *pc);

/*
 * Cache full blocks: index d_keys[i] -> d_block_ids[i] for i < count (device
 * arrays).  A key already present keeps its block id; if one call inserts
 * the same key twice with different ids, one of them is kept.  A key that
 * finds no free slot sets PKV_DEVERR_TABLE_FULL in d_error (optional device
 * int32) and is not cached.
 */
int pkv_prefix_cache_insert(pkv_prefix_cache *pc, const uint64_t *d_keys,
                            const int32_t *d_block_ids, int64_t count, int32_t *d_error,
                            pkv_stream_t s);

/*
 * Longest cached prefix of each of n requests (all arrays device memory):
 * request i's keys are d_keys[d_offsets[i] .. d_offsets[i+1]); d_max_hits[i]
 * caps the hit (pass floor((num_tokens - 1) / block_size) so the last position
 * is always recomputed).  d_hit_blocks[i] receives the number of leading
 * blocks whose keys are all cached (at most the cap), and d_hit_ids the cached
 * block ids of those blocks, -1 for the rest of the request's keys.  Up to
 * PKV_MAX_BATCH requests, every key of the batch below its request's cap is
 * probed by its own thread and each request keeps its first miss (three
 * launches); larger batches take one CTA per request.
 */
int pkv_prefix_cache_match(pkv_prefix_cache *pc, const uint64_t *d_keys, const int32_t *d_offsets,
                           const int32_t *d_max_hits, int32_t n, int32_t *d_hit_blocks,
                           int32_t *d_hit_ids, pkv_stream_t s);

/* ------------------------------------------------------------------------ */
/* Free-block pools and allocate_slots ("allocate_slots()" section of        */
/* "从源码读 vLLM Scheduler").                                               */
/* ------------------------------------------------------------------------ */

/* Set group `group`'s free-block stack to free_ids[0..count) (host array;
   the last entry is the top).  Ids must lie in [0, num_blocks). */
int pkv_pool_reset(pkv_state *st, int32_t group, const int32_t *free_ids, int32_t count,
                   pkv_stream_t s);

/* Number of free blocks on group `group`'s stack (host mirror, no wait). */
int pkv_pool_size(pkv_state *st, int32_t group, int32_t *count);

/* Synchronous: copy the bottom max_count entries of the stack to host ids. */
int pkv_pool_read(pkv_state *st, int32_t group, int32_t *ids, int32_t max_count,
                  pkv_stream_t s);

/*
 * Allocate the blocks a batch of scheduled requests needs, in order, as the
 * page's allocate_slots does for each request ("allocate_slots()" section of
 * "从源码读 vLLM Scheduler"): (1) slots needed = completed_tokens +
 * num_new_tokens[i] + num_lookahead[i] (NULL = 0); (2) per group, when
 * sliding_window[g] > 0 (host array [num_groups], NULL = no window), the held
 * blocks wholly before max(0, completed - (window - 1)) go onto the group's
 * free stack, lowest logical block first, and become -1 in the row;
 * (3) new blocks = needed - held; (4) the request is refused when
 * new + watermark_blocks exceeds the group's free blocks at that point
 * (which include the frees of step 2 of this and every earlier request of
 * the call); (5) otherwise its new ids are popped from the top of each
 * group's stack and appended to its table rows.  Each request goes through
 * all five steps before the next.  The first refused request (in any group)
 * and every later one are not admitted; the refused request's frees stand.
 * *out_admitted = how many were admitted; out_new_blocks (host
 * [n][num_groups], may be NULL) receives the new-block counts (0 for the
 * requests not admitted).  rows, num_new_tokens, num_lookahead: host [n].
 *
 * Steps (1)-(5) run on the GPU (three kernels on s: one CTA plans the whole
 * batch with a scan of the stack heights, then the pops and the pushes move
 * the ids).  Synchronous: the call waits for s and copies the admission
 * result back, because a scheduler acts on it at once.  The whole batch is
 * checked before anything changes.  Errors: PKV_ERR_NOT_ACTIVE;
 * PKV_ERR_INVALID_ARG (a row listed twice, a negative count, n above
 * PKV_MAX_BATCH, or (12 + 40 * num_groups) * n + 64 bytes above a quarter of
 * the state's pinned ring); PKV_ERR_CAPACITY (a request needing more blocks
 * than its table row holds, or a stack growing past its pool size) -- with
 * any error, no table entry or stack entry has changed.
 */
int pkv_allocate_slots(pkv_state *st, const int32_t *rows, const int32_t *num_new_tokens,
                       const int32_t *num_lookahead, int32_t n, const int32_t *sliding_window,
                       int32_t watermark_blocks, int32_t *out_admitted, int32_t *out_new_blocks,
                       pkv_stream_t s);

/*
 * Return the held blocks of rows[0..n) to their groups' stacks (in logical
 * order) and clear the table rows -- what happens to a finished request's
 * private blocks.  Blocks are not reference counted: a block shared between
 * requests must be released once.  PKV_ERR_CAPACITY if a stack would exceed
 * its pool size.
 */
int pkv_release_blocks(pkv_state *st, const int32_t *rows, int32_t n, pkv_stream_t s);

/* Synchronous: read the state's device error word into *code and clear it. */
int pkv_get_error(pkv_state *st, int32_t *code);

/* The state's device error word, for kv_cache_write's d_error. */
int pkv_state_error_word(pkv_state *st, int32_t **d_error);

/* Host-side view of one row: live flag, completed tokens, known token count
   and, when n_blocks is not NULL, blocks per group (host int32[num_groups]). */
int pkv_row_info(pkv_state *st, int32_t row, int32_t *active, int32_t *completed,
                 int32_t *n_tokens, int32_t *n_blocks);

/* Synchronous debug snapshot of one row's device data into host memory:
   completed_tokens, the first n_tokens token ids (tokens may be NULL), and
   each group's full block-table row (block_table[g] host int32[W_g], may be
   NULL). */
int pkv_read_row(pkv_state *st, int32_t row, int32_t *completed, int32_t *tokens,
                 int32_t n_tokens, int32_t *const *block_table, pkv_stream_t s);

/* The CUDA error code behind the last PKV_ERR_CUDA on this thread. */
int pkv_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * Self-test of the bounded waits inside the kernels (the prepare kernel's
 * wait for its staged schedule is one): launches one CTA of 32 threads whose
 * first thread waits on a shared-memory barrier that nothing completes, for
 * at most `polls` polls of at most 1 us each, then sets PKV_DEVERR_TIMEOUT
 * in *d_error (device int32, ORed in) and returns -- the same give-up path a
 * real wait takes, so a caller can check that it ends and reports.
 * polls: 1 .. 1000000.  Asynchronous on s.
 * Errors: PKV_ERR_INVALID_ARG (null d_error, polls out of range),
 * PKV_ERR_CUDA.
 */
int pkv_selftest_wait_timeout(int32_t *d_error, uint32_t polls, pkv_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
