/*
 * pkv_oracle.c -- CPU oracle for the per-step paged-KV input preparation.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library) never calls it, includes it or shares code with it.
 *
 * What it restates, as plain single-threaded loops over flat arrays:
 *
 *   - the worker's persistent request state (completed tokens, token ids,
 *     block table), kept per row of a pooled table whose rows are handed out
 *     on arrival and recycled on completion -- "Worker Request State
 *     Management" / "Design Logic Behind the Dual-Index System" on the page
 *     "Deep Dive into vLLM's Scheduling Mechanism: The Complete CPU-to-GPU
 *     Mapping Pipeline" (kongchang.com; its Chinese original is
 *     "vLLM调度机制深度解析", same sections);
 *   - batch construction: pick the scheduled rows, sort them by the number of
 *     tokens they run this step, record index_mapping ("Extracting the
 *     Execution Batch from Global State");
 *   - flattening: query_start_loc, positions, input_ids ("Contiguous Token
 *     Sequence Processing"); seq_lens ("Complete Input Preparation for the
 *     Attention Module");
 *   - the address chain position -> (logic_block, offset) -> physical block ->
 *     slot, per KV-cache group, and the gathered block tables ("Multi-Layer
 *     Coordinate Conversion Pipeline", "Address Calculation Example");
 *   - storing each new token's K and V vectors at its slot (same sections:
 *     a slot holds one token's K and V over all heads).
 *
 * Readings where the pages leave a step open (each is stated where used):
 *   R1  sort ascending by tokens this step; equal counts keep schedule order.
 *   R3  the null block id is -1; a scheduled position whose block is -1 or
 *       past the row's blocks is an error.
 *   R4  input_block_tables is the full block-table row (width W), -1 padded.
 *   R5  a new request takes the lowest free row; removal resets the row.
 *   R6  add_request takes the known token ids; update_request appends block
 *       ids and token ids and may set the computed-token count.
 *   R7  prepare reads completed_tokens as each request's start position; with
 *       the advance flag it then adds the scheduled count.
 *   R8  slot ids are 64-bit.
 *   R9  one cache line per slot per K (and per V): line_bytes contiguous bytes.
 *   R10 a negative slot is skipped by the KV store.
 *   R17 attention reads the first ceil(seq_len / bs) entries of a table row.
 *   R22 the paged (CSR) table lists those entries request after request.
 *
 * Status codes: 0 ok, 1 bad argument, 2 no free row, 3 row not active,
 * 4 capacity (positions, tokens or blocks missing).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MAX_GROUPS 8

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_FULL = 2, OR_NOT_ACTIVE = 3, OR_CAPACITY = 4 };

typedef struct {
    int32_t rows;
    int32_t max_len;
    int32_t G;
    int32_t bs[OR_MAX_GROUPS];
    int32_t W[OR_MAX_GROUPS];
    int64_t num_blocks[OR_MAX_GROUPS];
    uint8_t *active;      /* [rows] */
    int32_t *completed;   /* [rows] completed_tokens */
    int32_t *ntok;        /* [rows] how many token ids are known */
    int32_t **tok;        /* [rows] -> ntok[row] token ids */
    int32_t *nblk;        /* [G * rows] block ids held */
    int32_t *bt[OR_MAX_GROUPS]; /* [rows * W_g] block table, -1 where none */
    int32_t *pool[OR_MAX_GROUPS];   /* free block ids, a stack (allocate_slots) */
    int32_t pool_count[OR_MAX_GROUPS];
    int32_t pool_cap[OR_MAX_GROUPS];
} oracle_state;

/* ------------------------------------------------------------------------ */
/* state                                                                    */
/* ------------------------------------------------------------------------ */

void oracle_state_free(oracle_state *st)
{
    if (!st) return;
    if (st->tok)
        for (int32_t r = 0; r < st->rows; r++) free(st->tok[r]);
    free(st->tok);
    free(st->active);
    free(st->completed);
    free(st->ntok);
    free(st->nblk);
    for (int g = 0; g < OR_MAX_GROUPS; g++) {
        free(st->bt[g]);
        free(st->pool[g]);
    }
    free(st);
}

oracle_state *oracle_state_new(int32_t rows, int32_t max_len, int32_t G,
                               const int32_t *block_size, const int32_t *max_blocks,
                               const int64_t *num_blocks)
{
    if (rows <= 0 || max_len <= 0 || G <= 0 || G > OR_MAX_GROUPS) return NULL;
    oracle_state *st = (oracle_state *)calloc(1, sizeof(oracle_state));
    if (!st) return NULL;
    st->rows = rows;
    st->max_len = max_len;
    st->G = G;
    st->active = (uint8_t *)calloc((size_t)rows, 1);
    st->completed = (int32_t *)calloc((size_t)rows, sizeof(int32_t));
    st->ntok = (int32_t *)calloc((size_t)rows, sizeof(int32_t));
    st->tok = (int32_t **)calloc((size_t)rows, sizeof(int32_t *));
    st->nblk = (int32_t *)calloc((size_t)rows * G, sizeof(int32_t));
    int ok = st->active && st->completed && st->ntok && st->tok && st->nblk;
    for (int g = 0; g < G && ok; g++) {
        if (block_size[g] <= 0 || max_blocks[g] <= 0 || num_blocks[g] <= 0) { ok = 0; break; }
        st->bs[g] = block_size[g];
        st->W[g] = max_blocks[g];
        st->num_blocks[g] = num_blocks[g];
        st->bt[g] = (int32_t *)malloc((size_t)rows * max_blocks[g] * sizeof(int32_t));
        if (!st->bt[g]) { ok = 0; break; }
        for (int64_t k = 0; k < (int64_t)rows * max_blocks[g]; k++) st->bt[g][k] = -1;
    }
    if (!ok) { oracle_state_free(st); return NULL; }
    return st;
}

/* A block id is either a physical block of the group's pool or the null id. */
static int block_id_ok(const oracle_state *st, int g, int32_t id)
{
    return id == -1 || (id >= 0 && (int64_t)id < st->num_blocks[g]);
}

/* Append token ids to a row (R6). */
static int append_tokens(oracle_state *st, int32_t row, const int32_t *ids, int32_t n)
{
    if (n == 0) return OR_OK;
    int32_t old = st->ntok[row];
    int32_t *p = (int32_t *)realloc(st->tok[row], (size_t)(old + n) * sizeof(int32_t));
    if (!p) return OR_BAD_ARG;
    for (int32_t k = 0; k < n; k++) p[old + k] = ids[k];
    st->tok[row] = p;
    st->ntok[row] = old + n;
    return OR_OK;
}

/*
 * add_request: a new request gets a row and its state (completed tokens,
 * token ids, block ids) -- "add_request(): initialise state and block_table
 * for a new request" (Worker Request State Management).  The row is the
 * lowest free one (R5).  block_ids is the concatenation of the G groups'
 * lists, n_blocks[g] ids each.
 */
int oracle_add_request(oracle_state *st, const int32_t *token_ids, int32_t n_tokens,
                       int32_t num_computed, const int32_t *block_ids,
                       const int32_t *n_blocks, int32_t *out_row)
{
    if (n_tokens < 0 || n_tokens > st->max_len) return OR_BAD_ARG;
    if (num_computed < 0 || num_computed > n_tokens) return OR_BAD_ARG;
    int64_t off = 0;
    for (int g = 0; g < st->G; g++) {
        if (n_blocks[g] < 0 || n_blocks[g] > st->W[g]) return OR_BAD_ARG;
        for (int32_t j = 0; j < n_blocks[g]; j++)
            if (!block_id_ok(st, g, block_ids[off + j])) return OR_BAD_ARG;
        off += n_blocks[g];
    }
    int32_t row = -1;
    for (int32_t r = 0; r < st->rows; r++)
        if (!st->active[r]) { row = r; break; }
    if (row < 0) return OR_FULL;

    st->active[row] = 1;
    st->completed[row] = num_computed;
    st->ntok[row] = 0;
    free(st->tok[row]);
    st->tok[row] = NULL;
    if (append_tokens(st, row, token_ids, n_tokens) != OR_OK) return OR_BAD_ARG;
    off = 0;
    for (int g = 0; g < st->G; g++) {
        int32_t *line = st->bt[g] + (int64_t)row * st->W[g];
        for (int32_t j = 0; j < st->W[g]; j++)
            line[j] = j < n_blocks[g] ? block_ids[off + j] : -1;
        st->nblk[(int64_t)g * st->rows + row] = n_blocks[g];
        off += n_blocks[g];
    }
    *out_row = row;
    return OR_OK;
}

/*
 * update_request: "append newly allocated block IDs for an already registered
 * request" (Worker Request State Management), plus newly known token ids and,
 * when num_computed >= 0, the computed-token count the scheduler reports (R6).
 */
int oracle_update_request(oracle_state *st, int32_t row, const int32_t *new_block_ids,
                          const int32_t *n_new_blocks, const int32_t *new_token_ids,
                          int32_t n_new_tokens, int32_t num_computed)
{
    if (row < 0 || row >= st->rows) return OR_BAD_ARG;
    if (!st->active[row]) return OR_NOT_ACTIVE;
    if (n_new_tokens < 0) return OR_BAD_ARG;
    if ((int64_t)st->ntok[row] + n_new_tokens > st->max_len) return OR_CAPACITY;
    int64_t off = 0;
    for (int g = 0; g < st->G; g++) {
        int32_t have = st->nblk[(int64_t)g * st->rows + row];
        if (n_new_blocks[g] < 0) return OR_BAD_ARG;
        if (have + n_new_blocks[g] > st->W[g]) return OR_CAPACITY;
        for (int32_t j = 0; j < n_new_blocks[g]; j++)
            if (!block_id_ok(st, g, new_block_ids[off + j])) return OR_BAD_ARG;
        off += n_new_blocks[g];
    }
    if (num_computed > st->ntok[row] + n_new_tokens) return OR_BAD_ARG;

    off = 0;
    for (int g = 0; g < st->G; g++) {
        int32_t *line = st->bt[g] + (int64_t)row * st->W[g];
        int32_t have = st->nblk[(int64_t)g * st->rows + row];
        for (int32_t j = 0; j < n_new_blocks[g]; j++) line[have + j] = new_block_ids[off + j];
        st->nblk[(int64_t)g * st->rows + row] = have + n_new_blocks[g];
        off += n_new_blocks[g];
    }
    if (append_tokens(st, row, new_token_ids, n_new_tokens) != OR_OK) return OR_BAD_ARG;
    if (num_computed >= 0) st->completed[row] = num_computed;
    return OR_OK;
}

/* A finished request gives its row back for reuse; the row is reset (R5). */
int oracle_remove_request(oracle_state *st, int32_t row)
{
    if (row < 0 || row >= st->rows) return OR_BAD_ARG;
    if (!st->active[row]) return OR_NOT_ACTIVE;
    st->active[row] = 0;
    st->completed[row] = 0;
    for (int g = 0; g < st->G; g++) {
        int32_t *line = st->bt[g] + (int64_t)row * st->W[g];
        for (int32_t j = 0; j < st->W[g]; j++) line[j] = -1;
        st->nblk[(int64_t)g * st->rows + row] = 0;
    }
    return OR_OK;
}

/* Read back one row: its flags, counters, token ids and block-table lines. */
int oracle_read_row(const oracle_state *st, int32_t row, int32_t *active, int32_t *completed,
                    int32_t *ntok, int32_t *tokens_out, int32_t *nblk_out, int32_t *bt_out)
{
    if (row < 0 || row >= st->rows) return OR_BAD_ARG;
    *active = st->active[row];
    *completed = st->completed[row];
    *ntok = st->ntok[row];
    if (tokens_out)
        for (int32_t k = 0; k < st->ntok[row]; k++) tokens_out[k] = st->tok[row][k];
    int64_t off = 0;
    for (int g = 0; g < st->G; g++) {
        if (nblk_out) nblk_out[g] = st->nblk[(int64_t)g * st->rows + row];
        if (bt_out)
            for (int32_t j = 0; j < st->W[g]; j++)
                bt_out[off + j] = st->bt[g][(int64_t)row * st->W[g] + j];
        off += st->W[g];
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* batch construction                                                       */
/* ------------------------------------------------------------------------ */

/*
 * "Sort by the number of tokens to execute in this round" (Extracting the
 * Execution Batch from Global State).  R1: ascending, ties in schedule order.
 * Plain insertion sort, which is stable.
 */
static void sort_by_scheduled(const int32_t *num_sched, int32_t n, int32_t *order)
{
    for (int32_t i = 0; i < n; i++) order[i] = i;
    for (int32_t i = 1; i < n; i++) {
        int32_t cur = order[i];
        int32_t k = i - 1;
        while (k >= 0 && num_sched[order[k]] > num_sched[cur]) {
            order[k + 1] = order[k];
            k--;
        }
        order[k + 1] = cur;
    }
}

/*
 * One step's batch.  Inputs: the scheduled rows and their token counts in
 * schedule-output order.  Outputs (caller-allocated, n requests, T tokens):
 *   index_mapping[n], query_start_loc[n+1], seq_lens[n], positions[T],
 *   input_ids[T], and per group g: block_tables[g] ([n][W_g]) and
 *   slot_mapping[g] ([T], int64).
 * Everything is validated before any output is written.
 */
int oracle_prepare_batch(oracle_state *st, const int32_t *rows, const int32_t *num_sched,
                         int32_t n, int32_t advance,
                         int32_t *index_mapping, int32_t *query_start_loc,
                         int32_t *seq_lens, int32_t *positions, int32_t *input_ids,
                         int32_t *const *block_tables, int64_t *const *slot_mapping,
                         int32_t *out_total_tokens)
{
    if (n < 0) return OR_BAD_ARG;
    /* validation: every scheduled row is a live request, listed once, with
       token ids and block ids for every position it runs this step */
    int64_t total = 0;
    for (int32_t i = 0; i < n; i++) {
        int32_t r = rows[i];
        if (r < 0 || r >= st->rows) return OR_BAD_ARG;
        if (!st->active[r]) return OR_NOT_ACTIVE;
        if (num_sched[i] < 1) return OR_BAD_ARG;
        for (int32_t k = 0; k < i; k++)
            if (rows[k] == r) return OR_BAD_ARG;
        int64_t end = (int64_t)st->completed[r] + num_sched[i];
        if (end > st->ntok[r] || end > st->max_len) return OR_CAPACITY;
        for (int64_t p = st->completed[r]; p < end; p++)
            for (int g = 0; g < st->G; g++) {
                int64_t lb = p / st->bs[g];
                if (lb >= st->nblk[(int64_t)g * st->rows + r]) return OR_CAPACITY;
                if (st->bt[g][(int64_t)r * st->W[g] + lb] < 0) return OR_CAPACITY;
            }
        total += num_sched[i];
    }
    if (total > INT32_MAX) return OR_BAD_ARG;

    int32_t *order = (int32_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int32_t));
    int32_t *nb = (int32_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int32_t));
    if (!order || !nb) { free(order); free(nb); return OR_BAD_ARG; }

    /* batch_index -> request_state_index */
    sort_by_scheduled(num_sched, n, order);
    for (int32_t b = 0; b < n; b++) {
        index_mapping[b] = rows[order[b]];
        nb[b] = num_sched[order[b]];
    }

    /* query_start_loc: where each request's tokens start in the flat sequence
       (prefix-sum / CSR encoding, "Contiguous Token Sequence Processing") */
    query_start_loc[0] = 0;
    for (int32_t b = 0; b < n; b++) query_start_loc[b + 1] = query_start_loc[b] + nb[b];

    /* seq_lens: history plus this step's tokens */
    for (int32_t b = 0; b < n; b++) seq_lens[b] = st->completed[index_mapping[b]] + nb[b];

    /* per token: position, token id, and per group the write slot */
    for (int32_t b = 0; b < n; b++) {
        int32_t r = index_mapping[b];
        for (int32_t k = 0; k < nb[b]; k++) {
            int32_t t = query_start_loc[b] + k;           /* flat_token_index */
            int32_t p = st->completed[r] + k;              /* position */
            positions[t] = p;
            input_ids[t] = st->tok[r][p];
            for (int g = 0; g < st->G; g++) {
                int32_t bsz = st->bs[g];
                int32_t logic_block = p / bsz;             /* division */
                int32_t offset = p % bsz;                  /* remainder */
                int32_t physical = st->bt[g][(int64_t)r * st->W[g] + logic_block];
                slot_mapping[g][t] = (int64_t)physical * bsz + offset;
            }
        }
    }

    /* input_block_tables: each batch row's block-table row (R4) */
    for (int g = 0; g < st->G; g++)
        for (int32_t b = 0; b < n; b++)
            for (int32_t j = 0; j < st->W[g]; j++)
                block_tables[g][(int64_t)b * st->W[g] + j] =
                    st->bt[g][(int64_t)index_mapping[b] * st->W[g] + j];

    /* R7: optional advance of completed_tokens */
    if (advance)
        for (int32_t b = 0; b < n; b++) st->completed[index_mapping[b]] += nb[b];

    *out_total_tokens = (int32_t)total;
    free(order);
    free(nb);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* paged (CSR) block tables                                                 */
/* ------------------------------------------------------------------------ */

/*
 * The block-table entries attention reads, in paged CSR form.  "Complete
 * Input Preparation for the Attention Module": the block tables and seq_lens
 * together tell attention which physical blocks hold each request's KV and
 * how far its history reaches.  R17: request b reads the first
 * ceil(seq_lens[b] / bs) entries of its row.  R22: those entries are listed
 * one request after another in batch order (kv_indices); kv_indptr[b] is where
 * request b's list starts, an exclusive prefix sum like query_start_loc
 * ("Contiguous Token Sequence Processing"), kv_indptr[n] the total; and
 * last_page_len[b] counts the positions in the last listed block,
 * seq_lens[b] - (pages - 1) * bs.  index_mapping and seq_lens are a prepared
 * batch's outputs.  last_page_len may be NULL.  Returns OR_BAD_ARG, writing
 * nothing, for a row that is not live, seq_lens[b] < 1, more pages than the
 * row has entries (W_g), or more than capacity entries in all.
 */
int oracle_kv_indices(const oracle_state *st, int32_t g, const int32_t *index_mapping,
                      const int32_t *seq_lens, int32_t n, int32_t *kv_indptr,
                      int32_t *kv_indices, int64_t capacity, int32_t *last_page_len)
{
    if (g < 0 || g >= st->G || n < 0) return OR_BAD_ARG;
    int32_t bsz = st->bs[g];
    int64_t total = 0;
    for (int32_t b = 0; b < n; b++) {
        int32_t r = index_mapping[b];
        if (r < 0 || r >= st->rows || !st->active[r]) return OR_BAD_ARG;
        if (seq_lens[b] < 1) return OR_BAD_ARG;
        int64_t pages = ((int64_t)seq_lens[b] + bsz - 1) / bsz;   /* ceil */
        if (pages > st->W[g]) return OR_BAD_ARG;
        total += pages;
    }
    if (total > capacity || total > INT32_MAX) return OR_BAD_ARG;

    kv_indptr[0] = 0;
    for (int32_t b = 0; b < n; b++) {
        int32_t r = index_mapping[b];
        int32_t pages = (int32_t)(((int64_t)seq_lens[b] + bsz - 1) / bsz);
        kv_indptr[b + 1] = kv_indptr[b] + pages;
        for (int32_t j = 0; j < pages; j++)
            kv_indices[kv_indptr[b] + j] = st->bt[g][(int64_t)r * st->W[g] + j];
        if (last_page_len) last_page_len[b] = seq_lens[b] - (pages - 1) * bsz;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* KV store                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * "slot_mapping marks the write slots for this round's new tokens" and a slot
 * stores one token's K and V vectors over all heads (Multi-Layer Coordinate
 * Conversion Pipeline).  R9: k_cache and v_cache are arrays of num_slots lines
 * of line_bytes each; token t's K line starts at k + t*k_stride_bytes.
 * R10: negative slots are skipped.  Returns OR_BAD_ARG (writing nothing) if
 * any slot is at or beyond num_slots.
 */
int oracle_kv_write(const uint8_t *k, const uint8_t *v, int64_t k_stride_bytes,
                    int64_t v_stride_bytes, uint8_t *k_cache, uint8_t *v_cache,
                    int64_t num_slots, int32_t line_bytes, const int64_t *slot_mapping,
                    int32_t num_tokens)
{
    if (num_tokens < 0 || line_bytes <= 0) return OR_BAD_ARG;
    for (int32_t t = 0; t < num_tokens; t++)
        if (slot_mapping[t] >= num_slots) return OR_BAD_ARG;
    for (int32_t t = 0; t < num_tokens; t++) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        memcpy(k_cache + s * line_bytes, k + (int64_t)t * k_stride_bytes, (size_t)line_bytes);
        memcpy(v_cache + s * line_bytes, v + (int64_t)t * v_stride_bytes, (size_t)line_bytes);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* prefix-cache block keys                                                  */
/* ------------------------------------------------------------------------ */

/*
 * "Prefix Cache" section of "从源码读 vLLM Scheduler": what is hashed is a
 * token block together with its prefix context (not the K/V tensors); the hash
 * only indexes the cache, and a hit reuses the block's K/V; hits are limited
 * to num_tokens - 1 so the last position is always recomputed.  The page does
 * not fix the hash function.  Reading R18:
 *   digest_j = FNV-1a 64 over the 4*bs little-endian bytes of block j's ids
 *   key_j    = key_{j-1} * FNV_PRIME + digest_j  (mod 2^64),
 *              key_{-1} = FNV offset basis
 * so key_j depends on blocks 0..j in order.
 */
#define OR_FNV_BASIS 0xcbf29ce484222325ULL
#define OR_FNV_PRIME 0x00000100000001b3ULL

uint64_t oracle_fnv1a64(const uint8_t *bytes, int64_t len)
{
    uint64_t h = OR_FNV_BASIS;
    for (int64_t i = 0; i < len; i++) {
        h ^= bytes[i];
        h *= OR_FNV_PRIME;
    }
    return h;
}

/* Keys of the full blocks of token_ids[0..n_tokens): floor(n/bs) of them. */
int oracle_block_keys(const int32_t *token_ids, int32_t n_tokens, int32_t block_size,
                      uint64_t *keys)
{
    if (block_size <= 0 || n_tokens < 0) return OR_BAD_ARG;
    uint64_t prev = OR_FNV_BASIS;
    int32_t nfull = n_tokens / block_size;
    uint8_t *buf = (uint8_t *)malloc((size_t)block_size * 4);
    if (!buf) return OR_BAD_ARG;
    for (int32_t j = 0; j < nfull; j++) {
        for (int32_t k = 0; k < block_size; k++) {
            uint32_t t = (uint32_t)token_ids[(int64_t)j * block_size + k];
            buf[4 * k + 0] = (uint8_t)(t & 0xff);
            buf[4 * k + 1] = (uint8_t)((t >> 8) & 0xff);
            buf[4 * k + 2] = (uint8_t)((t >> 16) & 0xff);
            buf[4 * k + 3] = (uint8_t)((t >> 24) & 0xff);
        }
        uint64_t digest = oracle_fnv1a64(buf, (int64_t)block_size * 4);
        prev = prev * OR_FNV_PRIME + digest;
        keys[j] = prev;
    }
    free(buf);
    return OR_OK;
}

/* Keys of the full blocks of a row of the oracle state. */
int oracle_row_block_keys(const oracle_state *st, int32_t row, int32_t block_size,
                          uint64_t *keys, int32_t *n_keys)
{
    if (row < 0 || row >= st->rows || !st->active[row]) return OR_NOT_ACTIVE;
    *n_keys = st->ntok[row] / block_size;
    return oracle_block_keys(st->tok[row], st->ntok[row], block_size, keys);
}

/*
 * Longest prefix hit against an index of cached (key, block id) pairs: the
 * largest k <= floor((n_tokens - 1) / bs) with keys 0..k-1 all cached (R19:
 * only blocks wholly inside the first n_tokens - 1 positions can hit).  Fills
 * hit_ids[0..k) with the cached block ids.  The index is a plain array,
 * searched linearly.
 */
int32_t oracle_prefix_hits(const uint64_t *keys, int32_t n_tokens, int32_t block_size,
                           const uint64_t *index_keys, const int32_t *index_ids,
                           int64_t index_len, int32_t *hit_ids)
{
    if (n_tokens <= 0) return 0;
    int32_t cap = (n_tokens - 1) / block_size;
    int32_t k = 0;
    for (; k < cap; k++) {
        int64_t found = -1;
        for (int64_t e = 0; e < index_len; e++)
            if (index_keys[e] == keys[k]) { found = e; break; }
        if (found < 0) break;
        hit_ids[k] = index_ids[found];
    }
    return k;
}

/* ------------------------------------------------------------------------ */
/* block pool and allocate_slots                                            */
/* ------------------------------------------------------------------------ */

/*
 * "allocate_slots()" section of "从源码读 vLLM Scheduler": for one request,
 * in this order: (1) count the slots needed from the computed tokens, the new
 * tokens and the speculative lookahead; (2) free the sliding-window blocks no
 * longer needed; (3) count the new blocks actually missing; (4) keep a
 * watermark in reserve and check that enough free blocks remain -- available
 * = free - reserved, required = new + watermark, refuse if required >
 * available; (5) allocate.  A refused request is not scheduled; the scheduler
 * stops at it (it breaks out of its loop over waiting requests).
 *
 * Readings (R20): one call handles a batch of requests one after the other,
 * each through steps (1)-(5) before the next one starts; the first request
 * refused in any group, and every request after it, is not admitted; a
 * refused request's window frees (step 2, which comes before the check)
 * stand; "reserved" is 0 (nothing else holds blocks aside); each group's free
 * blocks form a stack: frees are pushed on top lowest logical block first,
 * and an allocation takes ids from the top, one at a time (so a request's own
 * frees can serve it).  Blocks wholly before max(0, computed - (window - 1))
 * are out of the window.  The whole batch is checked (rows live and distinct,
 * every request fits its table rows) before anything changes.
 */
int oracle_pool_reset(oracle_state *st, int32_t g, const int32_t *ids, int32_t count)
{
    if (g < 0 || g >= st->G || count < 0) return OR_BAD_ARG;
    free(st->pool[g]);
    st->pool_cap[g] = count + 16;
    st->pool[g] = (int32_t *)malloc((size_t)st->pool_cap[g] * sizeof(int32_t));
    if (!st->pool[g]) return OR_BAD_ARG;
    for (int32_t k = 0; k < count; k++) st->pool[g][k] = ids[k];
    st->pool_count[g] = count;
    return OR_OK;
}

int32_t oracle_pool_count(const oracle_state *st, int32_t g) { return st->pool_count[g]; }

void oracle_pool_read(const oracle_state *st, int32_t g, int32_t *out)
{
    for (int32_t k = 0; k < st->pool_count[g]; k++) out[k] = st->pool[g][k];
}

static void pool_push(oracle_state *st, int32_t g, int32_t id)
{
    if (st->pool_count[g] == st->pool_cap[g]) {
        st->pool_cap[g] = st->pool_cap[g] * 2 + 16;
        st->pool[g] = (int32_t *)realloc(st->pool[g], (size_t)st->pool_cap[g] * sizeof(int32_t));
    }
    st->pool[g][st->pool_count[g]++] = id;
}

/* Step (1): the slots a request needs once this step's tokens (and the
   speculative lookahead) are placed: computed tokens + new + lookahead. */
static int64_t slots_needed(const oracle_state *st, int32_t r, int32_t num_new, int32_t lookahead)
{
    return (int64_t)st->completed[r] + num_new + lookahead;
}

/* Step (2) for row r: push every held block wholly before
   max(0, computed - (window - 1)) onto its group's stack, lowest logical
   block first, and clear it from the row. */
static void free_out_of_window(oracle_state *st, int32_t r, const int32_t *window)
{
    for (int g = 0; g < st->G; g++) {
        if (window[g] <= 0) continue;
        int32_t *line = st->bt[g] + (int64_t)r * st->W[g];
        int32_t have = st->nblk[(int64_t)g * st->rows + r];
        int64_t start = (int64_t)st->completed[r] - (window[g] - 1);
        if (start < 0) start = 0;
        int32_t to = (int32_t)(start / st->bs[g]);
        if (to > have) to = have;
        for (int32_t j = 0; j < to; j++) {
            if (line[j] < 0) continue;   /* freed earlier */
            pool_push(st, g, line[j]);
            line[j] = -1;
        }
    }
}

int oracle_allocate_slots(oracle_state *st, const int32_t *rows, const int32_t *num_new,
                          const int32_t *lookahead, int32_t n, const int32_t *window,
                          int32_t watermark, int32_t *out_admitted, int32_t *out_new_blocks)
{
    /* the whole batch is checked first */
    for (int32_t i = 0; i < n; i++) {
        int32_t r = rows[i];
        if (r < 0 || r >= st->rows || !st->active[r]) return OR_NOT_ACTIVE;
        if (num_new[i] < 0 || (lookahead && lookahead[i] < 0)) return OR_BAD_ARG;
        for (int32_t k = 0; k < i; k++)
            if (rows[k] == r) return OR_BAD_ARG;
        int64_t need_len = slots_needed(st, r, num_new[i], lookahead ? lookahead[i] : 0);
        for (int g = 0; g < st->G; g++)
            if ((need_len + st->bs[g] - 1) / st->bs[g] > st->W[g]) return OR_CAPACITY;
    }
    int32_t admitted = n;
    for (int32_t i = 0; i < n; i++) {
        int32_t r = rows[i];
        /* (1) slots needed */
        int64_t need_len = slots_needed(st, r, num_new[i], lookahead ? lookahead[i] : 0);
        /* (2) free the blocks wholly out of the window */
        if (window) free_out_of_window(st, r, window);
        /* (3) new blocks missing; (4) watermark check */
        int32_t new_blocks[OR_MAX_GROUPS];
        int refused = 0;
        for (int g = 0; g < st->G; g++) {
            int32_t have = st->nblk[(int64_t)g * st->rows + r];
            int32_t need = (int32_t)((need_len + st->bs[g] - 1) / st->bs[g]);
            new_blocks[g] = need > have ? need - have : 0;
            int32_t available = st->pool_count[g] - 0;   /* reserved = 0 */
            if (new_blocks[g] + watermark > available) refused = 1;
        }
        if (refused) { admitted = i; break; }
        /* (5) allocate: take ids from the top of each stack */
        for (int g = 0; g < st->G; g++) {
            int32_t *line = st->bt[g] + (int64_t)r * st->W[g];
            int32_t have = st->nblk[(int64_t)g * st->rows + r];
            for (int32_t k = 0; k < new_blocks[g]; k++) {
                st->pool_count[g]--;
                line[have + k] = st->pool[g][st->pool_count[g]];
            }
            st->nblk[(int64_t)g * st->rows + r] = have + new_blocks[g];
            if (out_new_blocks) out_new_blocks[i * st->G + g] = new_blocks[g];
        }
    }
    for (int32_t i = admitted; i < n && out_new_blocks; i++)
        for (int g = 0; g < st->G; g++) out_new_blocks[i * st->G + g] = 0;
    *out_admitted = admitted;
    return OR_OK;
}

/*
 * A finished request's blocks go back to its groups' pools (pushed in
 * logical order, held blocks only) and its table rows are cleared.  Blocks
 * shared between requests are not reference counted: release each once.
 */
int oracle_release_blocks(oracle_state *st, const int32_t *rows, int32_t n)
{
    for (int32_t i = 0; i < n; i++) {
        int32_t r = rows[i];
        if (r < 0 || r >= st->rows || !st->active[r]) return OR_NOT_ACTIVE;
        for (int g = 0; g < st->G; g++) {
            int32_t *line = st->bt[g] + (int64_t)r * st->W[g];
            int32_t have = st->nblk[(int64_t)g * st->rows + r];
            for (int32_t j = 0; j < have; j++) {
                if (line[j] >= 0) pool_push(st, g, line[j]);
                line[j] = -1;
            }
            st->nblk[(int64_t)g * st->rows + r] = 0;
        }
    }
    return OR_OK;
}
