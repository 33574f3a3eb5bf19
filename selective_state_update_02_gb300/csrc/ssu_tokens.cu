// Multi-token decode step for GB300 (sm_103a): T consecutive tokens of every request in one
// call (the verification step of multi-token speculation, vLLM PR #48110, Test Plan).  Token t
// applies the single-token update to the state token t - 1 left; the state is loaded once,
// kept in registers (fp32) across the T tokens, and stored once.  Templated like the VEC
// kernel (rows per warp, columns per lane with dstate = 32 * NC, state type, index type), with
// its element mapping, update order and readout tree, so T = 1 reproduces ssu_update bit for
// bit.  Each warp prefetches token t + 1's inputs (dt, its NC columns of B and C, one x row per
// lane) while it updates token t.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ssu.h"
#include "ssu_device.cuh"
#include "ssu_host.h"

using ssu_host::aligned;
using ssu_host::DeviceGuard;
using ssu_host::fail;
using ssu_host::ok;
using ssu_host::validate_impl;

namespace {

struct TokenParams {
    SsuParams p;
    void *inter;                       // optional intermediate states (state dtype), may be null
    long long x_t, out_t, dt_t, B_t, C_t;
    long long in_b, in_t, in_h, in_p;  // intermediate strides; dstate stride is 1
    int tokens;
};

// update_lane (ssu_device.cuh) with the state update in packed fp32x2 instructions (two IEEE round-to-nearest
// multiplies and two fused multiply-adds per pair of columns): the same values bit for bit,
// with half the instructions for the update.  The readout chain stays scalar, in the same
// order.  Used where instruction issue, not memory, bounds the kernel (the multi-token loop).
template <int NC>
__device__ __forceinline__ float update_lane_packed(float (&v)[NC], float dA, float k,
                                                    const float (&bb)[NC], const float (&cc)[NC]) {
    const float2 dA2 = make_float2(dA, dA), k2 = make_float2(k, k);
#pragma unroll
    for (int j = 0; j < NC; j += 2) {
        const float2 kb = __fmul2_rn(k2, make_float2(bb[j], bb[j + 1]));
        const float2 r = __ffma2_rn(make_float2(v[j], v[j + 1]), dA2, kb);
        v[j] = r.x;
        v[j + 1] = r.y;
    }
    float part = v[0] * cc[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) part = fmaf(v[j], cc[j], part);
    return part;
}

// One token's inputs for one warp: lane r < RPW holds x of row r.
template <int NC>
struct TokenIn {
    float dt;
    float bb[NC], cc[NC];
    float x;
};

template <int RPW, int NC>
__device__ __forceinline__ TokenIn<NC> load_token(const TokenParams &q, long long b, int h,
                                                  int g, int row0, int t, int lane) {
    const SsuParams &p = q.p;
    TokenIn<NC> in;
    in.dt = __bfloat162float(p.dt[b * p.dt_b + t * q.dt_t + h * p.dt_h]);
    load_bc<NC>(p.B + b * p.B_b + t * q.B_t + g * p.B_g + lane_offset<NC>(lane), in.bb);
    load_bc<NC>(p.C + b * p.C_b + t * q.C_t + g * p.C_g + lane_offset<NC>(lane), in.cc);
    in.x = (lane < RPW && row0 + lane < p.headdim)
               ? __bfloat162float(p.x[b * p.x_b + t * q.x_t + h * p.x_h + row0 + lane])
               : 0.f;
    return in;
}

// 16 rows per warp hold 64 state values per lane: those CTAs are limited to 4 warps so the
// compiler may use up to 255 registers without spilling.
template <int RPW>
constexpr int tokens_max_threads() {
    return RPW >= 16 ? 128 : 32 * kMaxWarpsPerCta;
}

template <int RPW, int NC, typename ST, bool kIdx64>
__global__ void __launch_bounds__(tokens_max_threads<RPW>())
    ssu_tokens_kernel(const __grid_constant__ TokenParams q) {
    pdl_wait();
    const SsuParams &p = q.p;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int slab = blockIdx.x;
    const int h = blockIdx.y;
    for (long long b = blockIdx.z; b < p.batch; b += gridDim.z) {
        const long long s = load_slot<kIdx64>(p, b);
        if (s < 0 || s >= p.pool_size) {
            if (h == 0 && slab == 0 && threadIdx.x == 0) record_skip(p, b);
            continue;
        }
        const int row0 = slab * p.rows_per_cta + warp * RPW;
        ST *srow = static_cast<ST *>(p.state) + s * p.st_pool + h * p.st_head +
                   row0 * p.st_row + lane_offset<NC>(lane);

        float v[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (row0 + r < p.headdim) {
                load_cols<NC, ST>(srow + r * p.st_row, v[r]);
            } else {
#pragma unroll
                for (int j = 0; j < NC; ++j) v[r][j] = 0.f;
            }
        }

        const float bias = p.dt_bias[h * p.bias_h];
        const float Ah = p.A[h * p.A_h];
        const float Dh = p.D[h * p.D_h];
        const int g = h / p.heads_per_group;
        TokenIn<NC> cur = load_token<RPW, NC>(q, b, h, g, row0, 0, lane);
        for (int t = 0; t < q.tokens; ++t) {
            TokenIn<NC> nxt = cur;
            if (t + 1 < q.tokens) nxt = load_token<RPW, NC>(q, b, h, g, row0, t + 1, lane);
            const float dtv = softplus_f32(cur.dt + bias);
            const float dA = expf(dtv * Ah);
            float part[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float xr = __shfl_sync(0xffffffffu, cur.x, r);
                part[r] = update_lane_packed<NC>(v[r], dA, dtv * xr, cur.bb, cur.cc);
            }
            if (q.inter) {
                ST *irow = static_cast<ST *>(q.inter) + b * q.in_b + t * q.in_t + h * q.in_h +
                           row0 * q.in_p + lane_offset<NC>(lane);
#pragma unroll
                for (int r = 0; r < RPW; ++r)
                    if (row0 + r < p.headdim) store_cols<NC, ST>(irow + r * q.in_p, v[r]);
            }
            const float total = reduce_rows<RPW>(part, lane);
            const int rl = row_of_lane<RPW>(lane);
            const float xr = __shfl_sync(0xffffffffu, cur.x, rl);
            if (writes_row<RPW>(lane) && row0 + rl < p.headdim)
                p.out[b * p.out_b + t * q.out_t + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
            cur = nxt;
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            if (row0 + r < p.headdim) store_cols<NC, ST>(srow + r * p.st_row, v[r]);
    }
    pdl_trigger();  // this CTA's stores are issued: a dependent launch may start its CTAs
}

template <int RPW, int NC, typename ST, bool kIdx64>
cudaError_t launch_tokens_one(const TokenParams &q, dim3 grid, dim3 block, bool pdl,
                              cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ssu_tokens_kernel<RPW, NC, ST, kIdx64>, q);
}

template <int NC, typename ST, bool kIdx64>
cudaError_t launch_tokens_t(const TokenParams &q, int rpw, int wpc, dim3 grid, bool pdl,
                            cudaStream_t st) {
    const dim3 block(32 * wpc);
    switch (rpw) {
        case 1: return launch_tokens_one<1, NC, ST, kIdx64>(q, grid, block, pdl, st);
        case 2: return launch_tokens_one<2, NC, ST, kIdx64>(q, grid, block, pdl, st);
        case 4: return launch_tokens_one<4, NC, ST, kIdx64>(q, grid, block, pdl, st);
        case 8: return launch_tokens_one<8, NC, ST, kIdx64>(q, grid, block, pdl, st);
        case 16:
            if constexpr (NC <= 4)
                return static_cast<int>(block.x) <= tokens_max_threads<16>()
                           ? launch_tokens_one<16, NC, ST, kIdx64>(q, grid, block, pdl, st)
                           : cudaErrorInvalidValue;
            else
                return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tokens(const TokenParams &q, int nc, bool bf16, bool i64, int rpw, int wpc,
                          dim3 grid, bool pdl, cudaStream_t st) {
#define SSU_TOK_NC(NC_)                                                                      \
    if (nc == NC_) {                                                                         \
        if (bf16)                                                                            \
            return i64 ? launch_tokens_t<NC_, __nv_bfloat16, true>(q, rpw, wpc, grid, pdl, st) \
                       : launch_tokens_t<NC_, __nv_bfloat16, false>(q, rpw, wpc, grid, pdl,    \
                                                                    st);                       \
        return i64 ? launch_tokens_t<NC_, float, true>(q, rpw, wpc, grid, pdl, st)             \
                   : launch_tokens_t<NC_, float, false>(q, rpw, wpc, grid, pdl, st);           \
    }
    SSU_TOK_NC(2)
    SSU_TOK_NC(4)
    SSU_TOK_NC(8)
#undef SSU_TOK_NC
    return cudaErrorInvalidValue;
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
    const ssu_shape_t &s = *shape;
    // 8 rows per warp, one warp per CTA (fewer rows for a small headdim), or the handle's VEC
    // override for sweeps (16 rows per warp for dstate up to 128).
    int rpw = 8;
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

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                    static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535));
    const cudaError_t e = launch_tokens(q, static_cast<int>(s.dstate / 32),
                                        s.state_dtype == SSU_STATE_BF16,
                                        s.index_dtype == SSU_INDEX_I64, rpw, wpc, grid,
                                        handle->pdl, cs);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ok();
}
