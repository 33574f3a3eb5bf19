// Multi-token decode step: the C entry point ssu_update_tokens (validation, launch shape) and
// the kernels' instantiations; the kernel itself is in ssu_tokens.cuh.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ssu.h"
#include "ssu_host.h"
#include "ssu_tokens.cuh"
#include "ssu_tokens_mma.cuh"

using ssu_host::aligned;
using ssu_host::DeviceGuard;
using ssu_host::fail;
using ssu_host::ok;
using ssu_host::validate_impl;

namespace {

template <int N, typename ST, bool kIdx64>
cudaError_t launch_tokens_t(const TokenParams &q, dim3 grid, int rpw, int warps, bool pdl,
                            cudaStream_t st) {
    constexpr int RPI = RowGeo<N, ST>::RPI;
    constexpr int PD = token_prefetch<N, ST>();
#define SSU_TOK(R_) launch_tokens_one<R_, N, ST, kIdx64, PD>(q, grid, warps, pdl, st)
    if (rpw == RPI) return SSU_TOK(RPI);
    if (rpw == 2 * RPI) return SSU_TOK(2 * RPI);
    if (rpw == 4 * RPI) return SSU_TOK(4 * RPI);
    if (rpw == 8 * RPI) return SSU_TOK(8 * RPI);
    if constexpr (N == 128 && sizeof(ST) == 4)
        if (rpw == 16) return SSU_TOK(16);
#undef SSU_TOK
    return cudaErrorInvalidValue;
}

cudaError_t launch_tokens(const TokenParams &q, dim3 grid, int dstate, bool bf16, bool i64,
                          int rpw, int warps, bool pdl, cudaStream_t st) {
#define SSU_TOK_N(N_)                                                                         \
    if (dstate == N_) {                                                                       \
        if (bf16)                                                                             \
            return i64 ? launch_tokens_t<N_, __nv_bfloat16, true>(q, grid, rpw, warps, pdl, st) \
                       : launch_tokens_t<N_, __nv_bfloat16, false>(q, grid, rpw, warps, pdl, st); \
        return i64 ? launch_tokens_t<N_, float, true>(q, grid, rpw, warps, pdl, st)             \
                   : launch_tokens_t<N_, float, false>(q, grid, rpw, warps, pdl, st);           \
    }
    SSU_TOK_N(64)
    SSU_TOK_N(128)
    SSU_TOK_N(256)
#undef SSU_TOK_N
    return cudaErrorInvalidValue;
}

// The chunked kernel's instantiations: fp32 state at dstate 64 and 128, bf16 at 128 (a bf16
// state at dstate 64 never takes it, see mma_min_tokens).
cudaError_t launch_mma(const TokenParams &q, dim3 grid, int dstate, bool bf16, bool i64,
                       int warps, bool pdl, cudaStream_t st) {
    if (bf16) {
        if (dstate != 128) return cudaErrorInvalidValue;
        return i64 ? launch_tokens_mma<128, __nv_bfloat16, true>(q, grid, warps, pdl, st)
                   : launch_tokens_mma<128, __nv_bfloat16, false>(q, grid, warps, pdl, st);
    }
    if (dstate == 64)
        return i64 ? launch_tokens_mma<64, float, true>(q, grid, warps, pdl, st)
                   : launch_tokens_mma<64, float, false>(q, grid, warps, pdl, st);
    if (dstate == 128)
        return i64 ? launch_tokens_mma<128, float, true>(q, grid, warps, pdl, st)
                   : launch_tokens_mma<128, float, false>(q, grid, warps, pdl, st);
    return cudaErrorInvalidValue;
}

// The chunked matrix-form kernel (ssu_tokens_mma.cuh) takes a call without intermediate
// states and without a launch override when dstate is 64 or 128, headdim is a multiple of 8,
// B, C and x can be staged in 16-byte pieces (base addresses 16-byte aligned, every stride a
// multiple of 8 elements) and the call has at least mma_min_tokens tokens.  Its work per tile
// hardly depends on T (up to 8 tokens per chunk), the general kernel's grows with T; the
// crossovers measured at batch 128, 16 heads (us per call, general / chunked):
//   fp32 dstate 128: T 4: 28.7 / 29.3, T 6: 35.1 / 30.6, T 8: 40.2 / 31.5, T 16: 63.6 / 43.9
//   fp32 dstate 64:  T 4: 15.7 / 17.7, T 6: 18.9 / 18.2, T 8: 22.5 / 18.6, T 16: 35.8 / 27.4
//   bf16 dstate 128: T 4: 20.3 / 29.1, T 8: 30.5 / 31.5, T 16: 49.2 / 46.6
//   bf16 dstate 64:  T 4: 12.6 / 17.8, T 8: 18.3 / 20.1, T 16: 28.1 / 30.2
// (a bf16 state halves the general kernel's bytes, not the chunked kernel's arithmetic).
int mma_min_tokens(int64_t dstate, int32_t state_dtype) {
    if (state_dtype != SSU_STATE_BF16) return 5;
    return dstate == 128 ? 16 : SSU_MAX_TOKENS + 1;
}

bool mma_eligible(const ssu_shape_t &s, const ssu_strides_t &str, const ssu_token_strides_t &ts,
                  const void *x, const void *B, const void *C, int64_t tokens) {
    if (s.dstate != 64 && s.dstate != 128) return false;
    if (tokens < mma_min_tokens(s.dstate, s.state_dtype)) return false;
    if (s.headdim % 8 != 0) return false;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16)) return false;
    const long long strides[] = {str.x[0], str.x[1], ts.x, str.B[0], str.B[1], ts.B,
                                 str.C[0], str.C[1], ts.C};
    for (long long v : strides)
        if (v % 8 != 0) return false;
    return true;
}

}  // namespace

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
    const bool use_mma = !intermediate && !handle->has_override &&
                         mma_eligible(s, *strides, *ts, x, B, C, tokens);
    // From the sweeps (bench.py --tokens --sweep, batch 128, T = 2 and 4, every bucket): an fp32
    // state takes 32 fp32 values per lane (8 vector rows at 4 columns per lane, 4 at 8 for
    // dstate 256), a bf16 state 64 (8 vector rows at 8 columns: 2, 4 or 8 rows per vector
    // row), in CTAs of 2 warps; bf16 dstate 128 at T = 2 / 4: 19.45 / 25.52 us with 4 vector
    // rows, 16.16 / 20.67 with 8; fp32 dstate 128: 24.30 / 29.33 at 1 warp per CTA, 23.87 /
    // 29.14 at 2.  Fewer rows for a small headdim.  The handle's VEC override (for sweeps) sets
    // rows per warp and warps per CTA instead.
    const int rpi = ssu_host::rows_per_instruction(s.dstate, s.state_dtype);
    const long long row_bytes = s.dstate * (s.state_dtype == SSU_STATE_BF16 ? 2 : 4);
    const int vpr = row_bytes >= 512 ? static_cast<int>(row_bytes / 512) : 1;  // vectors per lane
    const int nc = (s.state_dtype == SSU_STATE_BF16 ? 8 : 4) * vpr;            // columns per lane
    int slots = (s.state_dtype == SSU_STATE_BF16 ? 64 : 32) / nc;
    while (slots > 1 && slots * rpi > s.headdim) slots >>= 1;
    int rpw = slots * rpi;
    int wpc = 2;
    while (wpc > 1 && rpw * wpc > s.headdim) wpc >>= 1;
    if (handle->has_override && handle->override_launch.mode == SSU_MODE_VEC) {
        rpw = handle->override_launch.rows_per_warp;
        wpc = handle->override_launch.warps_per_cta;
        if (!ssu_host::rows_per_warp_ok(rpw, s.dstate, s.state_dtype))
            return fail(SSU_ERR_UNSUPPORTED, "%d rows per warp do not fit dstate %lld", rpw,
                        (long long)s.dstate);
        if ((rpw / rpi) * nc > 64 || ((rpw / rpi) * nc > 32 && wpc > 4))
            return fail(SSU_ERR_UNSUPPORTED,
                        "the multi-token kernel holds at most 64 state values per lane (32 in "
                        "CTAs of more than 4 warps)");
    }
    if (use_mma) {  // 16 rows per warp, up to 4 warps (64 rows) per CTA
        rpw = kMmaRowsPerWarp;
        wpc = kMmaWarpsPerCta;
        while (wpc > 1 && rpw * (wpc / 2) >= s.headdim) wpc >>= 1;
    }
    const long long slabs = (s.headdim + rpw * wpc - 1) / (rpw * wpc);
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
    p.rows_per_cta = rpw * wpc;
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
    // multiple of the 16-byte vector's elements: 4 for an fp32 state, 8 for bf16) is 8-byte
    // (16-byte) aligned at every request, token and group.
    {
        const int epv = s.state_dtype == SSU_STATE_BF16 ? 8 : 4;
        const bool b_ok = aligned(B, 2 * epv) && strides->B[0] % epv == 0 &&
                          strides->B[1] % epv == 0 && ts->B % epv == 0;
        const bool c_ok = aligned(C, 2 * epv) && strides->C[0] % epv == 0 &&
                          strides->C[1] % epv == 0 && ts->C % epv == 0;
        q.bc_vec = b_ok && c_ok;
    }

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16 = s.state_dtype == SSU_STATE_BF16, i64 = s.index_dtype == SSU_INDEX_I64;
    const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                    static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535));
    const cudaError_t e =
        use_mma ? launch_mma(q, grid, static_cast<int>(s.dstate), bf16, i64, wpc, handle->pdl, cs)
                : launch_tokens(q, grid, static_cast<int>(s.dstate), bf16, i64, rpw, wpc,
                                handle->pdl, cs);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ok();
}
