/*
 * One decode step driven from plain C99 through include/ssu.h: the boundary needs no C++ and
 * no torch.  Device memory comes from the CUDA runtime's C API, which is the caller's job (the
 * library allocates nothing for an update).
 *
 * The case is the hand-computed one of the oracle's pins, widened to dstate 64 with zero
 * columns: S = [1, 2, 0, ...], x = 1, dt = dt_bias = 0, A = -1, B = [1, -1, 0, ...],
 * C = [1, 1, 0, ...], D = 0.5, so dtv = ln 2, dA = 1/2, S' = [0.5 + ln 2, 1 - ln 2, 0, ...] and
 * y = 2 exactly (bf16 0x4000).  A second pool slot must stay untouched.  The step then runs
 * again from the same pool through ssu_update_from_host with the per-step operands and the
 * readout in page-locked host memory, and must give the same bits.
 *
 * Exit status 0 and "ok" on success; "no-device" (status 0) when no GPU is present, after the
 * host-side checks; a message and status 1 otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ssu.h"

#define N 64

static int fail(const char *what) {
    printf("FAIL: %s (%s)\n", what, ssu_last_error());
    return 1;
}

int main(void) {
    ssu_shape_t shape;
    ssu_strides_t st;
    memset(&shape, 0, sizeof shape);
    memset(&st, 0, sizeof st);
    shape.batch = 1;
    shape.nheads = 1;
    shape.headdim = 1;
    shape.dstate = N;
    shape.ngroups = 1;
    shape.pool_size = 2;
    shape.index_dtype = SSU_INDEX_I32;
    shape.state_dtype = SSU_STATE_F32;
    st.state[0] = N, st.state[1] = N, st.state[2] = N, st.state[3] = 1;
    st.x[0] = 1, st.x[1] = 1, st.x[2] = 1;
    st.out[0] = 1, st.out[1] = 1, st.out[2] = 1;
    st.dt[0] = 1, st.dt[1] = 1, st.dt[2] = 0;
    st.B[0] = N, st.B[1] = N, st.B[2] = 1;
    st.C[0] = N, st.C[1] = N, st.C[2] = 1;
    st.dt_bias[0] = 1, st.dt_bias[1] = 0;
    st.D[0] = 1, st.D[1] = 0;
    st.A[0] = 1, st.A[1] = 0, st.A[2] = 0;
    st.idx = 1;

    if (ssu_abi_version() != SSU_ABI_VERSION) return fail("ABI version");
    if (strcmp(ssu_status_string(SSU_ERR_MISALIGNED), "SSU_ERR_MISALIGNED") != 0)
        return fail("status string");
    /* host-side validation with placeholder addresses (never dereferenced) */
    {
        char *fake = (char *)(uintptr_t)4096;
        if (ssu_validate(fake, fake, (const uint16_t *)fake, (const uint16_t *)fake,
                         (const float *)fake, (const float *)fake, (const uint16_t *)fake,
                         (const uint16_t *)fake, (const float *)fake, (const uint16_t *)fake,
                         &shape, &st) != SSU_OK)
            return fail("validate");
        shape.dstate = 96;
        if (ssu_validate(fake, fake, (const uint16_t *)fake, (const uint16_t *)fake,
                         (const float *)fake, (const float *)fake, (const uint16_t *)fake,
                         (const uint16_t *)fake, (const float *)fake, (const uint16_t *)fake,
                         &shape, &st) != SSU_ERR_UNSUPPORTED)
            return fail("dstate 96 must be unsupported");
        shape.dstate = N;
    }

    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count < 1) {
        ssu_handle_t h = NULL;
        if (ssu_create(&h, 0) != SSU_ERR_CUDA) return fail("create without a device");
        printf("no-device\n");
        return 0;
    }

    float pool[2 * N];
    memset(pool, 0, sizeof pool);
    pool[N + 0] = 1.0f; /* slot 1 is the request's; slot 0 must not change */
    pool[N + 1] = 2.0f;
    pool[0] = 7.0f;
    uint16_t B[N], C[N];
    memset(B, 0, sizeof B);
    memset(C, 0, sizeof C);
    B[0] = 0x3F80, B[1] = 0xBF80; /* 1, -1 */
    C[0] = 0x3F80, C[1] = 0x3F80; /* 1, 1 */
    const uint16_t x = 0x3F80, dt = 0x0000;
    const float dt_bias = 0.0f, A = -1.0f, D = 0.5f;
    const int idx = 1;

    float *d_pool, *d_bias, *d_A, *d_D;
    uint16_t *d_B, *d_C, *d_x, *d_dt, *d_out;
    int *d_idx;
    if (cudaMalloc((void **)&d_pool, sizeof pool) || cudaMalloc((void **)&d_B, sizeof B) ||
        cudaMalloc((void **)&d_C, sizeof C) || cudaMalloc((void **)&d_x, 2) ||
        cudaMalloc((void **)&d_dt, 2) || cudaMalloc((void **)&d_out, 2) ||
        cudaMalloc((void **)&d_bias, 4) || cudaMalloc((void **)&d_A, 4) ||
        cudaMalloc((void **)&d_D, 4) || cudaMalloc((void **)&d_idx, 4))
        return fail("cudaMalloc");
    cudaMemcpy(d_pool, pool, sizeof pool, cudaMemcpyHostToDevice);
    cudaMemcpy(d_B, B, sizeof B, cudaMemcpyHostToDevice);
    cudaMemcpy(d_C, C, sizeof C, cudaMemcpyHostToDevice);
    cudaMemcpy(d_x, &x, 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d_dt, &dt, 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d_bias, &dt_bias, 4, cudaMemcpyHostToDevice);
    cudaMemcpy(d_A, &A, 4, cudaMemcpyHostToDevice);
    cudaMemcpy(d_D, &D, 4, cudaMemcpyHostToDevice);
    cudaMemcpy(d_idx, &idx, 4, cudaMemcpyHostToDevice);

    ssu_handle_t h = NULL;
    if (ssu_create(&h, 0) != SSU_OK) return fail("create");
    if (ssu_update(h, d_pool, d_idx, d_x, d_dt, d_bias, d_A, d_B, d_C, d_D, d_out, &shape, &st,
                   NULL) != SSU_OK)
        return fail("update");
    uint32_t skipped = 99;
    int64_t first = 99;
    if (ssu_get_error(h, NULL, &skipped, &first) != SSU_OK || skipped != 0 || first != -1)
        return fail("error counters");
    uint16_t y = 0;
    float got[2 * N];
    cudaMemcpy(&y, d_out, 2, cudaMemcpyDeviceToHost);
    cudaMemcpy(got, d_pool, sizeof got, cudaMemcpyDeviceToHost);

    /* The same step with the per-step operands and the readout in page-locked host memory
       (ssu_update_from_host), from the original pool: the same bits. */
    {
        int *h_idx;
        uint16_t *h_x, *h_dt, *h_B, *h_C, *h_out;
        void *d_ws;
        int64_t ws_bytes = 0;
        if (cudaHostAlloc((void **)&h_idx, 4, cudaHostAllocDefault) ||
            cudaHostAlloc((void **)&h_x, 2, cudaHostAllocDefault) ||
            cudaHostAlloc((void **)&h_dt, 2, cudaHostAllocDefault) ||
            cudaHostAlloc((void **)&h_B, sizeof B, cudaHostAllocDefault) ||
            cudaHostAlloc((void **)&h_C, sizeof C, cudaHostAllocDefault) ||
            cudaHostAlloc((void **)&h_out, 2, cudaHostAllocDefault))
            return fail("cudaHostAlloc");
        *h_idx = idx, *h_x = x, *h_dt = dt, *h_out = 0xFFFF;
        memcpy(h_B, B, sizeof B);
        memcpy(h_C, C, sizeof C);
        if (ssu_host_workspace_bytes(&shape, &ws_bytes) != SSU_OK || ws_bytes < 256)
            return fail("workspace size");
        if (cudaMalloc(&d_ws, (size_t)ws_bytes)) return fail("cudaMalloc workspace");
        float *d_pool2;
        if (cudaMalloc((void **)&d_pool2, sizeof pool)) return fail("cudaMalloc pool");
        cudaMemcpy(d_pool2, pool, sizeof pool, cudaMemcpyHostToDevice);
        /* pageable host memory is refused before anything is enqueued */
        if (ssu_update_from_host(h, d_pool2, h_idx, h_x, h_dt, d_bias, d_A, B, h_C, d_D, h_out,
                                 &shape, &st, d_ws, ws_bytes, NULL) != SSU_ERR_INVALID_ARG)
            return fail("pageable B must be refused");
        if (ssu_update_from_host(h, d_pool2, h_idx, h_x, h_dt, d_bias, d_A, h_B, h_C, d_D, h_out,
                                 &shape, &st, d_ws, ws_bytes, NULL) != SSU_OK)
            return fail("update_from_host");
        if (cudaStreamSynchronize(NULL) != cudaSuccess) return fail("synchronize");
        float got2[2 * N];
        cudaMemcpy(got2, d_pool2, sizeof got2, cudaMemcpyDeviceToHost);
        if (*h_out != y) return fail("host-path readout differs");
        if (memcmp(got2, got, sizeof got) != 0) return fail("host-path state differs");
        cudaFree(d_pool2);
        cudaFree(d_ws);
        cudaFreeHost(h_idx), cudaFreeHost(h_x), cudaFreeHost(h_dt);
        cudaFreeHost(h_B), cudaFreeHost(h_C), cudaFreeHost(h_out);
    }
    ssu_destroy(h);

    const double ln2 = log(2.0);
    if (y != 0x4000) {
        printf("FAIL: readout bits 0x%04x, expected 0x4000 (2.0)\n", y);
        return 1;
    }
    if (fabs(got[N + 0] - (0.5 + ln2)) > 1e-5 * 2.2 || fabs(got[N + 1] - (1.0 - ln2)) > 1e-5 * 1.4)
        return fail("updated state");
    for (int n = 2; n < N; ++n)
        if (got[N + n] != 0.0f) return fail("zero columns must stay zero");
    if (got[0] != 7.0f) return fail("untouched slot changed");
    for (int n = 1; n < N; ++n)
        if (got[n] != 0.0f) return fail("untouched slot changed");
    printf("ok\n");
    return 0;
}
