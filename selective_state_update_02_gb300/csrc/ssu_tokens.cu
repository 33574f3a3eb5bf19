// Multi-token decode step: the C entry point ssu_update_tokens (validation, launch shape) and
// the kernels' instantiations; the kernel itself is in ssu_tokens.cuh.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ssu.h"
#include "ssu_host.h"
#include "ssu_tokens.cuh"

using ssu_host::aligned;
using ssu_host::DeviceGuard;
using ssu_host::fail;
using ssu_host::ok;
using ssu_host::validate_impl;

extern "C" ssu_status_t ssu_update_tokens(ssu_handle_t handle, void *state_pool,
                                          const void *state_batch_indices, const uint16_t *x,
                                          const uint16_t *dt, const float *dt_bias,
                                          const float *A, const uint16_t *B, const uint16_t *C,
                                          const float *D, uint16_t *out, void *intermediate,
                                          const ssu_shape_t *shape, const ssu_strides_t *strides,
                                          int64_t tokens, const ssu_token_strides_t *ts,
                                          ssu_stream_t stream) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    if (!ts) return fail(SSU_ERR_INVALID_ARG, "token strides must not be NULL");
    if (tokens < 1 || tokens > SSU_MAX_TOKENS)
        return fail(SSU_ERR_INVALID_ARG, "tokens %lld outside 1..%d", (long long)tokens,
                    SSU_MAX_TOKENS);
    ssu_status_t st = validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                                    D, out, shape, strides);
    if (st != SSU_OK || shape->batch == 0) return st;
    if (ts->x < 0 || ts->out < 0 || ts->dt < 0 || ts->B < 0 || ts->C < 0)
        return fail(SSU_ERR_INVALID_ARG, "negative token stride");
    if (intermediate) {
        for (int j = 0; j < 5; ++j)
            if (ts->intermediate[j] < 0) return fail(SSU_ERR_INVALID_ARG, "negative stride");
        if (ts->intermediate[4] != 1)
            return fail(SSU_ERR_UNSUPPORTED, "intermediate dstate-stride must be 1");
        const int per16 = shape->state_dtype == SSU_STATE_BF16 ? 8 : 4;
        for (int j = 0; j < 4; ++j)
            if (ts->intermediate[j] % per16)
                return fail(SSU_ERR_MISALIGNED,
                            "intermediate strides must be multiples of 16 bytes");
        if (!aligned(intermediate, 16))
            return fail(SSU_ERR_MISALIGNED, "intermediate is not 16-byte aligned");
    }
    // One token without intermediate states is the single step: it runs on ssu_update's
    // kernel, which gives the same bits (measured 22.6 against 23.2 us at batch 128).
    if (tokens == 1 && !intermediate)
        return ssu_update(handle, state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                          out, shape, strides, stream);
    const ssu_shape_t &s = *shape;
    // 8 rows per warp (4 at dstate 256), one warp per CTA (fewer rows for a small headdim), or
    // the handle's VEC override for sweeps (16 rows per warp for dstate up to 128).
    int rpw = s.dstate == 256 ? 4 : 8;
    while (rpw > 1 && rpw > s.headdim) rpw >>= 1;
    int wpc = 1;
    if (handle->has_override && handle->override_launch.mode == SSU_MODE_VEC) {
        rpw = handle->override_launch.rows_per_warp;
        wpc = handle->override_launch.warps_per_cta;
        if (rpw > 16 || (rpw == 16 && (s.dstate > 128 || wpc > 4)))
            return fail(SSU_ERR_UNSUPPORTED,
                        "the multi-token kernel takes 1..8 rows per warp (16 with at most 4 "
                        "warps, up to dstate 128)");
    }
    const int rows_per_tile = rpw * wpc;
    const long long slabs = (s.headdim + rows_per_tile - 1) / rows_per_tile;
    const long long tiles = s.batch * s.nheads * slabs;
    if (tiles > INT_MAX) return fail(SSU_ERR_UNSUPPORTED, "%lld tiles exceed 2^31", tiles);

    TokenParams q{};
    SsuParams &p = q.p;
    p.state = state_pool;
    p.idx = state_batch_indices;
    p.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    p.dt = reinterpret_cast<const __nv_bfloat16 *>(dt);
    p.dt_bias = dt_bias;
    p.A = A;
    p.B = reinterpret_cast<const __nv_bfloat16 *>(B);
    p.C = reinterpret_cast<const __nv_bfloat16 *>(C);
    p.D = D;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.st_pool = strides->state[0];
    p.st_head = strides->state[1];
    p.st_row = strides->state[2];
    p.x_b = strides->x[0];
    p.x_h = strides->x[1];
    p.out_b = strides->out[0];
    p.out_h = strides->out[1];
    p.dt_b = strides->dt[0];
    p.dt_h = strides->dt[1];
    p.B_b = strides->B[0];
    p.B_g = strides->B[1];
    p.C_b = strides->C[0];
    p.C_g = strides->C[1];
    p.bias_h = strides->dt_bias[0];
    p.D_h = strides->D[0];
    p.A_h = strides->A[0];
    p.idx_s = strides->idx;
    p.pool_size = s.pool_size;
    p.batch = s.batch;
    p.nheads = static_cast<int>(s.nheads);
    p.headdim = static_cast<int>(s.headdim);
    p.heads_per_group = static_cast<int>(s.nheads / s.ngroups);
    p.group_magic = group_magic(static_cast<unsigned>(p.heads_per_group));
    p.slabs = static_cast<int>(slabs);
    p.rows_per_cta = rows_per_tile;
    p.err = handle->err;
    q.inter = intermediate;
    q.x_t = ts->x;
    q.out_t = ts->out;
    q.dt_t = ts->dt;
    q.B_t = ts->B;
    q.C_t = ts->C;
    q.in_b = ts->intermediate[0];
    q.in_t = ts->intermediate[1];
    q.in_h = ts->intermediate[2];
    q.in_p = ts->intermediate[3];
    q.tokens = static_cast<int>(tokens);
    // Whole column groups of B and C are aligned vectors when the lane's first column (a
    // multiple of 4 columns, 2 at dstate 64) is 8-byte (4-byte) aligned at every request,
    // token and group.
    {
        const int pair = s.dstate == 64 ? 2 : 4;
        const bool b_ok = aligned(B, 2 * pair) && strides->B[0] % pair == 0 &&
                          strides->B[1] % pair == 0 && ts->B % pair == 0;
        const bool c_ok = aligned(C, 2 * pair) && strides->C[0] % pair == 0 &&
                          strides->C[1] % pair == 0 && ts->C % pair == 0;
        q.bc_vec = b_ok && c_ok;
    }

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                    static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535));
    const int nc = static_cast<int>(s.dstate / 32);
    const bool bf16 = s.state_dtype == SSU_STATE_BF16, i64 = s.index_dtype == SSU_INDEX_I64;
    const cudaError_t e = launch_tokens_depth<kTokenPrefetch>(q, nc, bf16, i64, rpw, wpc, grid,
                                                              handle->pdl, cs);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ok();
}
