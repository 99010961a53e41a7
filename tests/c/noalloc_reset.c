/*
 * kv_store_noalloc across a device reset, from plain C.  The entry point
 * keeps its static record's device address with the CUDA context it was
 * looked up in; cudaDeviceReset ends that context, and the next call, in the
 * new context, must look the address up again.  Each round allocates its
 * buffers, writes a batch with one out-of-range slot, and checks the cache
 * rows and the reported count and first bad token; between the rounds the
 * device is reset.  Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvstore.h"

#define T 6
#define H 2
#define D 16
#define SLOTS 32

static int fail(const char *what, int round)
{
    fprintf(stderr, "noalloc_reset: round %d: %s\n", round, what);
    return 1;
}

static int one_round(int round)
{
    const size_t row = H * D * sizeof(uint16_t);
    uint16_t k[T * H * D], v[T * H * D];
    for (int i = 0; i < T * H * D; ++i) {
        k[i] = (uint16_t)(0x3000 + 7 * round + i);
        v[i] = (uint16_t)(0x5000 + 11 * round + i);
    }
    /* token 3 is out of range in round 0, token 1 in round 1 */
    int32_t slots[T] = {4, 9, 31, 2, 17, 0};
    if (round == 0) slots[3] = SLOTS;
    else slots[1] = -7;
    void *dk, *dv, *dkc, *dvc, *didx;
    if (cudaMalloc(&dk, sizeof k) || cudaMalloc(&dv, sizeof v) || cudaMalloc(&dkc, SLOTS * row) ||
        cudaMalloc(&dvc, SLOTS * row) || cudaMalloc(&didx, sizeof slots))
        return fail("cudaMalloc", round);
    cudaMemcpy(dk, k, sizeof k, cudaMemcpyHostToDevice);
    cudaMemcpy(dv, v, sizeof v, cudaMemcpyHostToDevice);
    cudaMemcpy(didx, slots, sizeof slots, cudaMemcpyHostToDevice);
    cudaMemset(dkc, 0xEE, SLOTS * row);
    cudaMemset(dvc, 0xEE, SLOTS * row);
    const kv_strides s = {row, D * 2, 2, row, D * 2, 2, row, D * 2, 2, row, D * 2, 2};
    int64_t n_bad = -1, first_bad = -2;
    const kv_status st = kv_store_noalloc(dk, dv, dkc, dvc, didx, KV_INDEX_I32, 1, T, H, D, 2, &s,
                                          SLOTS, 0, &n_bad, &first_bad, NULL);
    if (st != KV_ERR_INDEX_OOB) return fail(kv_status_str(st), round);
    if (n_bad != 1 || first_bad != (round == 0 ? 3 : 1)) return fail("bad-slot report", round);
    uint16_t kc[SLOTS * H * D], vc[SLOTS * H * D];
    cudaMemcpy(kc, dkc, sizeof kc, cudaMemcpyDeviceToHost);
    cudaMemcpy(vc, dvc, sizeof vc, cudaMemcpyDeviceToHost);
    for (int t = 0; t < T; ++t) {
        if (slots[t] < 0 || slots[t] >= SLOTS) continue;
        if (memcmp(kc + slots[t] * H * D, k + t * H * D, row) ||
            memcmp(vc + slots[t] * H * D, v + t * H * D, row))
            return fail("row", round);
    }
    int written = 0;
    for (int slot = 0; slot < SLOTS; ++slot) {
        const uint8_t *b = (const uint8_t *)(kc + slot * H * D);
        int sentinel = 1;
        for (size_t i = 0; i < row; ++i) sentinel &= b[i] == 0xEE;
        written += !sentinel;
    }
    if (written != T - 1) return fail("stray rows", round);
    cudaFree(dk); cudaFree(dv); cudaFree(dkc); cudaFree(dvc); cudaFree(didx);
    return 0;
}

int main(void)
{
    if (one_round(0)) return 1;
    if (cudaDeviceReset() != cudaSuccess) return fail("cudaDeviceReset", 0);
    if (one_round(1)) return 1;
    printf("noalloc_reset: ok\n");
    return 0;
}
