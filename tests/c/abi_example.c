/*
 * A plain C caller of the KV-cache write library: no Python, no torch.
 * It allocates device memory with the CUDA runtime, writes a small batch
 * with kv_store and kv_store_fp8, reads the caches back and checks them
 * against the definitions (copy: the row lands at its slot byte for byte;
 * FP8: a few values with known e4m3fn codes), checks that an out-of-range
 * slot is reported by kv_error_poll and not written, gathers the copied
 * rows back with kv_gather, and writes one row with a per-token scale
 * computed in the kernel (kv_store_fp8_ex), checking the scale and codes.
 * Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvstore.h"

#define T 4
#define H 2
#define D 8
#define SLOTS 16

static int fail(const char *what)
{
    fprintf(stderr, "abi_example: %s\n", what);
    return 1;
}

int main(void)
{
    uint16_t k[T * H * D], v[T * H * D];
    for (int i = 0; i < T * H * D; ++i) {
        k[i] = (uint16_t)(0x1000 + i);
        v[i] = (uint16_t)(0x2000 + i);
    }
    int64_t slots[T] = {5, 0, 99, 12};           /* token 2 is out of range */
    const size_t row = H * D * sizeof(uint16_t);

    void *dk, *dv, *dkc, *dvc, *didx, *derr;
    if (cudaMalloc(&dk, sizeof k) || cudaMalloc(&dv, sizeof v) ||
        cudaMalloc(&dkc, SLOTS * row) || cudaMalloc(&dvc, SLOTS * row) ||
        cudaMalloc(&didx, sizeof slots) || cudaMalloc(&derr, sizeof(kv_error_record)))
        return fail("cudaMalloc");
    cudaMemcpy(dk, k, sizeof k, cudaMemcpyHostToDevice);
    cudaMemcpy(dv, v, sizeof v, cudaMemcpyHostToDevice);
    cudaMemcpy(didx, slots, sizeof slots, cudaMemcpyHostToDevice);
    cudaMemset(dkc, 0xEE, SLOTS * row);
    cudaMemset(dvc, 0xEE, SLOTS * row);
    cudaMemset(derr, 0, sizeof(kv_error_record));

    kv_strides s = {(int64_t)row, D * 2, 2, (int64_t)row, D * 2, 2,
                    (int64_t)row, D * 2, 2, (int64_t)row, D * 2, 2};
    kv_status st = kv_store(dk, dv, dkc, dvc, didx, KV_INDEX_I64, 1, T, H, D, 2, &s, SLOTS, 0,
                            (kv_error_record *)derr, NULL);
    if (st != KV_OK)
        return fail(kv_status_str(st));
    int64_t nbad = 0, first = 0;
    st = kv_error_poll((kv_error_record *)derr, NULL, &nbad, &first);
    if (st != KV_ERR_INDEX_OOB || nbad != 1 || first != 2)
        return fail("out-of-range slot not reported");

    uint16_t kc[SLOTS * H * D], vc[SLOTS * H * D];
    cudaMemcpy(kc, dkc, sizeof kc, cudaMemcpyDeviceToHost);
    cudaMemcpy(vc, dvc, sizeof vc, cudaMemcpyDeviceToHost);
    for (int t = 0; t < T; ++t) {
        if (slots[t] < 0 || slots[t] >= SLOTS)
            continue;
        if (memcmp(kc + slots[t] * H * D, k + t * H * D, row) ||
            memcmp(vc + slots[t] * H * D, v + t * H * D, row))
            return fail("copied row differs");
    }
    for (int slot = 0; slot < SLOTS; ++slot) {
        int named = 0;
        for (int t = 0; t < T; ++t)
            named |= slots[t] == slot;
        if (!named && kc[slot * H * D] != 0xEEEE)
            return fail("a slot nobody named was written");
    }

    /* FP8: bf16 1.0, -2.0, 448, 1e6 (saturates), 2^-9 with inv = 1 -> 0x38 0xC0 0x7E 0x7E 0x01 */
    uint16_t kb[T * H * D];
    const uint16_t vals[5] = {0x3F80, 0xC000, 0x43E0, 0x4974, 0x3B00};
    for (int i = 0; i < T * H * D; ++i)
        kb[i] = vals[i % 5];
    cudaMemcpy(dk, kb, sizeof kb, cudaMemcpyHostToDevice);
    int64_t ok_slots[T] = {1, 2, 3, 4};
    cudaMemcpy(didx, ok_slots, sizeof ok_slots, cudaMemcpyHostToDevice);
    uint8_t *dq;
    if (cudaMalloc((void **)&dq, 2 * SLOTS * H * D))
        return fail("cudaMalloc fp8");
    cudaMemset(dq, 0x7F, 2 * SLOTS * H * D);
    kv_strides s8 = {(int64_t)row, D * 2, 2, (int64_t)row, D * 2, 2,
                     H * D, D, 1, H * D, D, 1};
    st = kv_store_fp8(dk, dk, dq, dq + SLOTS * H * D, didx, KV_INDEX_I64, 1, T, H, D, KV_SRC_BF16,
                      &s8, 4, 4 * H * D, 4 * H * D, SLOTS, NULL, NULL, 0,
                      (kv_error_record *)derr, NULL);
    if (st != KV_OK)
        return fail(kv_status_str(st));
    if (kv_error_poll((kv_error_record *)derr, NULL, NULL, NULL) != KV_OK)
        return fail("fp8: unexpected error report");
    uint8_t q[SLOTS * H * D];
    cudaMemcpy(q, dq, sizeof q, cudaMemcpyDeviceToHost);
    const uint8_t want[5] = {0x38, 0xC0, 0x7E, 0x7E, 0x01};
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < H * D; ++e)
            if (q[ok_slots[t] * H * D + e] != want[(t * H * D + e) % 5])
                return fail("fp8 code differs");

    /* kv_gather: the rows of the in-range tokens come back byte for byte */
    uint16_t *dout;
    if (cudaMalloc((void **)&dout, 2 * sizeof k))
        return fail("cudaMalloc gather");
    cudaMemcpy(didx, slots, sizeof slots, cudaMemcpyHostToDevice);
    cudaMemset(dout, 0, 2 * sizeof k);
    st = kv_gather(dkc, dvc, dout, dout + T * H * D, didx, KV_INDEX_I64, 1, T, H, D, 2, &s,
                   SLOTS, (kv_error_record *)derr, NULL);
    if (st != KV_OK)
        return fail(kv_status_str(st));
    if (kv_error_poll((kv_error_record *)derr, NULL, &nbad, &first) != KV_ERR_INDEX_OOB ||
        nbad != 1 || first != 2)
        return fail("gather: out-of-range slot not reported");
    uint16_t back[2 * T * H * D];
    cudaMemcpy(back, dout, sizeof back, cudaMemcpyDeviceToHost);
    for (int t = 0; t < T; ++t) {
        if (t == 2)
            continue;
        if (memcmp(back + t * H * D, k + t * H * D, row) ||
            memcmp(back + T * H * D + t * H * D, v + t * H * D, row))
            return fail("gathered row differs");
    }

    /* kv_store_fp8_ex, one scale per token row: a row of 2.0 and -1.0 has
       amax 2, inv = 448/2 = 224, scale = 2/448, codes 0x7E and 0xF6 */
    uint16_t kd[T * H * D];
    for (int i = 0; i < T * H * D; ++i)
        kd[i] = (i % 2) ? 0xBF80 : 0x4000;          /* bf16 -1.0, 2.0 */
    cudaMemcpy(dk, kd, sizeof kd, cudaMemcpyHostToDevice);
    cudaMemcpy(didx, ok_slots, sizeof ok_slots, cudaMemcpyHostToDevice);
    float *dsc;
    if (cudaMalloc((void **)&dsc, 2 * SLOTS * sizeof(float)))
        return fail("cudaMalloc scales");
    cudaMemset(dq, 0x7F, 2 * SLOTS * H * D);
    st = kv_store_fp8_ex(dk, dk, dq, dq + SLOTS * H * D, didx, KV_INDEX_I64, 1, T, H, D,
                         KV_SRC_BF16, &s8, 4, 4 * H * D, 4 * H * D, SLOTS, KV_FP8_E4M3FN,
                         KV_SCALE_TOKEN, NULL, NULL, dsc, dsc + SLOTS, 1,
                         (kv_error_record *)derr, NULL);
    if (st != KV_OK)
        return fail(kv_status_str(st));
    if (kv_error_poll((kv_error_record *)derr, NULL, NULL, NULL) != KV_OK)
        return fail("fp8_ex: unexpected error report");
    float sc[2 * SLOTS];
    cudaMemcpy(q, dq, sizeof q, cudaMemcpyDeviceToHost);
    cudaMemcpy(sc, dsc, sizeof sc, cudaMemcpyDeviceToHost);
    const float want_scale = 2.0f / 448.0f;
    for (int t = 0; t < T; ++t) {
        if (sc[ok_slots[t]] != want_scale || sc[SLOTS + ok_slots[t]] != want_scale)
            return fail("fp8_ex: per-token scale differs");
        for (int e = 0; e < H * D; ++e)
            if (q[ok_slots[t] * H * D + e] != ((e % 2) ? 0xF6 : 0x7E))
                return fail("fp8_ex code differs");
    }
    cudaFree(dout);
    cudaFree(dsc);

    if (kv_abi_version() != KV_ABI_VERSION)
        return fail("ABI version");
    cudaFree(dk); cudaFree(dv); cudaFree(dkc); cudaFree(dvc); cudaFree(didx); cudaFree(derr);
    cudaFree(dq);
    printf("abi_example: ok\n");
    return 0;
}
