/*
 * The pages' worked example through the C ABI alone: plain C11, the CUDA
 * runtime for device memory, no Python and no PyTorch.  Request A (state row
 * 6, 16 computed tokens, blocks [81, 44]) runs 8 tokens and request B (row 7,
 * 31 computed tokens, blocks [37, 12]) runs 1 ("Design Logic Behind the
 * Dual-Index System", "Extracting the Execution Batch from Global State",
 * "Contiguous Token Sequence Processing" and "Address Calculation Example" on
 * "Deep Dive into vLLM's Scheduling Mechanism: The Complete CPU-to-GPU
 * Mapping Pipeline").  Exit status 0 and "ok" when every output matches.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pkv.h"

static int failures = 0;

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            failures++;                                                    \
        }                                                                  \
    } while (0)

#define CALL(expr)                                                         \
    do {                                                                   \
        int rc_ = (expr);                                                  \
        if (rc_ != PKV_OK) {                                               \
            fprintf(stderr, "%s:%d: %s returned %d\n", __FILE__, __LINE__, #expr, rc_); \
            return 1;                                                      \
        }                                                                  \
    } while (0)

static int same(const int32_t *a, const int32_t *b, int n) {
    return memcmp(a, b, (size_t)n * sizeof(int32_t)) == 0;
}

int main(void) {
    const int32_t bs = 16, W = 4;
    pkv_group_spec group = {bs, W, 1000};
    pkv_state *st = NULL;
    CALL(pkv_state_create(&st, 16, 64, 1, &group, 0, NULL));

    /* rows 0..7 taken, then 6 and 7 freed: A lands on 6, B on 7 */
    int32_t row = -1, none = 0;
    for (int i = 0; i < 8; i++) CALL(pkv_add_request(st, NULL, 0, 0, NULL, &none, &row, NULL));
    CALL(pkv_remove_request(st, 6, NULL));
    CALL(pkv_remove_request(st, 7, NULL));
    int32_t tok_a[24], tok_b[32];
    for (int p = 0; p < 24; p++) tok_a[p] = 6000 + p;
    for (int p = 0; p < 32; p++) tok_b[p] = 7000 + p;
    const int32_t blk_a[2] = {81, 44}, blk_b[2] = {37, 12}, two = 2;
    const int32_t *ba = blk_a, *bb = blk_b;
    CALL(pkv_add_request(st, tok_a, 24, 16, &ba, &two, &row, NULL));
    CHECK(row == 6);
    CALL(pkv_add_request(st, tok_b, 32, 31, &bb, &two, &row, NULL));
    CHECK(row == 7);

    /* the step: B with 1 token, A with 8, in schedule-output order */
    const int32_t rows[2] = {7, 6}, sched[2] = {1, 8};
    int32_t *d_i32 = NULL;
    int64_t *d_slots = NULL;
    if (cudaMalloc((void **)&d_i32, 64 * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc((void **)&d_slots, 16 * sizeof(int64_t)) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    pkv_batch_out out;
    memset(&out, 0, sizeof(out));
    out.index_mapping = d_i32;          /* [2] */
    out.query_start_loc = d_i32 + 2;    /* [3] */
    out.seq_lens = d_i32 + 5;           /* [2] */
    out.positions = d_i32 + 7;          /* [9] */
    out.input_ids = d_i32 + 16;         /* [9] */
    out.block_tables[0] = d_i32 + 28;   /* [2][4], 16-byte aligned */
    out.slot_mapping[0] = d_slots;      /* [9] */
    int32_t total = 0;
    CALL(pkv_prepare_batch(st, rows, sched, 2, 0, &out, &total, NULL));
    CHECK(total == 9);

    int32_t h[64];
    int64_t slots[9];
    cudaMemcpy(h, d_i32, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(slots, d_slots, sizeof(slots), cudaMemcpyDeviceToHost);
    const int32_t im[2] = {7, 6}, qsl[3] = {0, 1, 9}, sl[2] = {32, 24};
    const int32_t pos[9] = {31, 16, 17, 18, 19, 20, 21, 22, 23};
    const int32_t ids[9] = {7031, 6016, 6017, 6018, 6019, 6020, 6021, 6022, 6023};
    const int32_t tables[8] = {37, 12, -1, -1, 81, 44, -1, -1};
    CHECK(same(h, im, 2));
    CHECK(same(h + 2, qsl, 3));
    CHECK(same(h + 5, sl, 2));
    CHECK(same(h + 7, pos, 9));
    CHECK(same(h + 16, ids, 9));
    CHECK(same(h + 28, tables, 8));
    CHECK(slots[0] == 207);                       /* B: block 12, offset 15 */
    for (int t = 1; t < 9; t++) CHECK(slots[t] == 704 + (t - 1));   /* A: block 44 */

    /* the paged (CSR) view of the same batch */
    int32_t *d_csr = NULL;
    cudaMalloc((void **)&d_csr, 16 * sizeof(int32_t));
    CALL(pkv_kv_indices(st, 0, out.index_mapping, out.seq_lens, 2, d_csr, d_csr + 4, 8,
                        d_csr + 12, NULL));
    int32_t csr[16];
    cudaMemcpy(csr, d_csr, sizeof(csr), cudaMemcpyDeviceToHost);
    const int32_t indptr[3] = {0, 2, 4}, indices[4] = {37, 12, 81, 44}, last[2] = {16, 8};
    CHECK(same(csr, indptr, 3));
    CHECK(same(csr + 4, indices, 4));
    CHECK(same(csr + 12, last, 2));

    /* the KV store: 32-byte lines, token t's K line filled with t, V with 100 + t */
    enum { LINE = 32, SLOTS = 1000 * 16 };
    uint8_t hk[9 * LINE], hv[9 * LINE];
    for (int t = 0; t < 9; t++) {
        memset(hk + t * LINE, t, LINE);
        memset(hv + t * LINE, 100 + t, LINE);
    }
    uint8_t *dk = NULL, *dv = NULL, *kc = NULL, *vc = NULL;
    cudaMalloc((void **)&dk, sizeof(hk));
    cudaMalloc((void **)&dv, sizeof(hv));
    cudaMalloc((void **)&kc, (size_t)SLOTS * LINE);
    cudaMalloc((void **)&vc, (size_t)SLOTS * LINE);
    cudaMemset(kc, 0xEE, (size_t)SLOTS * LINE);
    cudaMemset(vc, 0xEE, (size_t)SLOTS * LINE);
    cudaMemcpy(dk, hk, sizeof(hk), cudaMemcpyHostToDevice);
    cudaMemcpy(dv, hv, sizeof(hv), cudaMemcpyHostToDevice);
    int32_t *d_error = NULL;
    CALL(pkv_state_error_word(st, &d_error));
    CALL(pkv_kv_cache_write(dk, dv, LINE, LINE, kc, vc, SLOTS, LINE, d_slots, 9, d_error, NULL));
    uint8_t line_k[LINE], line_v[LINE], untouched[LINE];
    for (int t = 0; t < 9; t++) {
        cudaMemcpy(line_k, kc + slots[t] * LINE, LINE, cudaMemcpyDeviceToHost);
        cudaMemcpy(line_v, vc + slots[t] * LINE, LINE, cudaMemcpyDeviceToHost);
        CHECK(memcmp(line_k, hk + t * LINE, LINE) == 0);
        CHECK(memcmp(line_v, hv + t * LINE, LINE) == 0);
    }
    cudaMemcpy(untouched, kc + 208 * LINE, LINE, cudaMemcpyDeviceToHost);
    for (int b = 0; b < LINE; b++) CHECK(untouched[b] == 0xEE);   /* slot 208: not written */

    int32_t code = -1;
    CALL(pkv_get_error(st, &code));
    CHECK(code == 0);
    CALL(pkv_state_destroy(st));
    cudaFree(d_i32);
    cudaFree(d_slots);
    cudaFree(d_csr);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(kc);
    cudaFree(vc);
    if (failures) {
        fprintf(stderr, "%d checks failed\n", failures);
        return 1;
    }
    printf("ok\n");
    return 0;
}
