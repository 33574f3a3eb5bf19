// Multi-token decode-step kernel for GB300 (sm_103a), instantiated by ssu_tokens.cu (which
// also holds the C entry point).
//
// The step: T consecutive tokens of every request in one
// call (the verification step of multi-token speculation, vLLM PR #48110, Test Plan).  Token t
// applies the single-token update to the state token t - 1 left; the state is loaded once,
// kept in registers (fp32) across the T tokens, and stored once.  Templated like the VEC
// kernel (rows per warp, columns per lane with dstate = 32 * NC, state type, index type), with
// its element mapping, update order and readout tree, so T = 1 reproduces ssu_update bit for
// bit.  Each warp keeps the inputs of the next tokens in flight (its NC columns of B and C and
// one x row per lane, as raw bf16 bits in a register ring) while it updates token t, and
// computes every token's dt and dA once per warp (lane j for token j, handed out by shuffles).

#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ssu_device.cuh"

namespace {

struct TokenParams {
    SsuParams p;
    void *inter;                       // optional intermediate states (state dtype), may be null
    long long x_t, out_t, dt_t, B_t, C_t;
    long long in_b, in_t, in_h, in_p;  // intermediate strides; dstate stride is 1
    int tokens;
    int bc_vec;  // B and C rows can be read as whole column pairs / quads (aligned vectors)
};

// update_lane (ssu_device.cuh) on one lane's NC columns held as fp32 pairs (column 2i in .x,
// 2i+1 in .y), the state update in packed fp32x2 instructions: two IEEE round-to-nearest
// multiplies and two fused multiply-adds per pair, so the same values bit for bit, with half
// the instructions.  The readout chain stays scalar, over the columns in the same order.
// Holding the state and B/C as pairs for the whole token loop saves the moves that form
// pairs out of scalar registers (measured 1-2 % faster at T >= 3).
template <int NC>
__device__ __forceinline__ float update_pairs(float2 (&w)[NC / 2], float2 dA2, float k,
                                              const float2 (&b2)[NC / 2],
                                              const float2 (&c2)[NC / 2]) {
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) w[i] = __ffma2_rn(w[i], dA2, __fmul2_rn(k2, b2[i]));
    float part = w[0].x * c2[0].x;
    part = fmaf(w[0].y, c2[0].y, part);
#pragma unroll
    for (int i = 1; i < NC / 2; ++i) {
        part = fmaf(w[i].x, c2[i].x, part);
        part = fmaf(w[i].y, c2[i].y, part);
    }
    return part;
}

// One token's inputs for one lane as raw bf16 bits: the lane's NC columns of B and C as column
// pairs (column 2i in the low half of word i, 2i+1 in the high half) and, in lanes r < RPW, x
// of row r.  They are widened to fp32 only where they are used, so the loads of later tokens
// stay in flight while earlier tokens are computed.
template <int NC>
struct TokenBits {
    unsigned b[NC / 2], c[NC / 2];
    unsigned short x;
};

// Tokens whose inputs a warp keeps in flight (the kernels' PD): the loads of token t + PD are
// issued as soon as token t's inputs have been widened.  A ring of 2, with the 8-row kernels
// up to dstate 128 held to 96 registers (tokens_max_regs below: 20 resident warps per SM, 5
// per sub-partition's register file, instead of 16 at 125 registers), measured faster than a
// ring of 4 without the cap at every token count, batch 128 (fp32 dstate 128, T = 2 / 3 / 4 /
// 8: 24.11 / 26.87 / 29.39 / 41.74 -> 23.99 / 26.01 / 28.70 / 40.26 us; fp32 dstate 64, T = 4:
// 22.07 -> 20.49; bf16 dstate 128, T = 4: 30.41 -> 26.79).  A ring of 3 at 104 registers was slower (T = 4: 30.50), a ring of 4
// spills under a cap of 112 or less, and a ring of 2 spills under 88.
constexpr int kTokenPrefetch = 2;

__device__ __forceinline__ float widen_bf16(unsigned short u) {
    return __uint_as_float(static_cast<unsigned>(u) << 16);  // exact: bf16 is fp32's top half
}

// Pair words widened to fp32 pairs.
template <int NC>
__device__ __forceinline__ void widen_pairs(const unsigned (&w)[NC / 2], float2 (&o)[NC / 2]) {
#pragma unroll
    for (int i = 0; i < NC / 2; ++i)
        o[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// The lane's NC columns starting at `p` (its first column) as pair words.  VEC: one 4- or
// 8-byte load per group of columns (the host checked the alignment); otherwise two 2-byte
// loads per pair.
template <int NC, bool VEC>
__device__ __forceinline__ void load_pairs(const unsigned short *p, unsigned (&w)[NC / 2]) {
    if constexpr (VEC) {
        if constexpr (NC == 2) {
            w[0] = *reinterpret_cast<const unsigned *>(p);
        } else {
#pragma unroll
            for (int g = 0; g < NC / 4; ++g) {
                const uint2 u = *reinterpret_cast<const uint2 *>(p + g * 128);
                w[2 * g] = u.x;
                w[2 * g + 1] = u.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
            const int j = 2 * i;
            const unsigned short *q = p + (j / 4) * 128 + (j % 4);
            w[i] = static_cast<unsigned>(q[0]) | (static_cast<unsigned>(q[1]) << 16);
        }
    }
}

// One token's inputs into a ring slot: `B` and `C` point at the lane's first column of the
// token's rows, `x` at the lane's x element (read only where `x_live`: lanes r < RPW whose row
// exists).
template <int NC, bool VEC>
__device__ __forceinline__ void load_token(const unsigned short *B, const unsigned short *C,
                                           const unsigned short *x, bool x_live,
                                           TokenBits<NC> &in) {
    load_pairs<NC, VEC>(B, in.b);
    load_pairs<NC, VEC>(C, in.c);
    in.x = x_live ? *x : static_cast<unsigned short>(0);
}

// dt and dA of token base + lane (lanes past the last token hold 0): each token's softplus
// and exponential are computed once per warp and handed out by shuffles.
__device__ __forceinline__ void token_scalars(const TokenParams &q, long long b, int h,
                                              float bias, float Ah, int base, int lane,
                                              float &dtv, float &dA) {
    const SsuParams &p = q.p;
    const int t = base + lane;
    dtv = 0.f;
    dA = 0.f;
    if (t < q.tokens) {
        const float z =
            widen_bf16(reinterpret_cast<const unsigned short *>(p.dt)[b * p.dt_b + t * q.dt_t +
                                                                      h * p.dt_h]) +
            bias;
        dtv = softplus_f32(z);
        dA = expf(dtv * Ah);
    }
}

// The T-token loop of one warp over its RPW rows held in v (see the kernel below).  The
// per-token inputs are read through pointers built once per warp and advanced by one token
// stride per token; the outputs' addresses are formed per token (carrying output pointers
// through the loop as well measured 5-10 % slower once the ring refills).
template <int RPW, int NC, typename ST, bool VEC, int PD>
__device__ __forceinline__ void token_loop(const TokenParams &q, float (&v)[RPW][NC], long long b,
                                           int h, int row0, int lane) {
    const SsuParams &p = q.p;
    const float bias = p.dt_bias[h * p.bias_h];
    const float Ah = p.A[h * p.A_h];
    const float Dh = p.D[h * p.D_h];
    const int g = group_of(h, p.group_magic);
    const int lo = lane_offset<NC>(lane);
    const unsigned short *Bn = reinterpret_cast<const unsigned short *>(p.B) + b * p.B_b +
                               g * p.B_g + lo;
    const unsigned short *Cn = reinterpret_cast<const unsigned short *>(p.C) + b * p.C_b +
                               g * p.C_g + lo;
    const bool x_live = lane < RPW && row0 + lane < p.headdim;
    const unsigned short *xn = reinterpret_cast<const unsigned short *>(p.x) + b * p.x_b +
                               h * p.x_h + row0 + (x_live ? lane : 0);
    // A ring of the next PD tokens' inputs, unrolled so every slot is a fixed register.
    TokenBits<NC> ring[PD];
#pragma unroll
    for (int k = 0; k < PD; ++k)
        if (k < q.tokens)
            load_token<NC, VEC>(Bn + k * q.B_t, Cn + k * q.C_t, xn + k * q.x_t, x_live, ring[k]);
    Bn += PD * q.B_t;  // now token PD's
    Cn += PD * q.C_t;
    xn += PD * q.x_t;
    float lane_dtv, lane_dA;
    token_scalars(q, b, h, bias, Ah, 0, lane, lane_dtv, lane_dA);
    float2 w[RPW][NC / 2];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) w[r][i] = make_float2(v[r][2 * i], v[r][2 * i + 1]);
    for (int t0 = 0; t0 < q.tokens; t0 += PD) {
#pragma unroll
        for (int k = 0; k < PD; ++k) {
            const int t = t0 + k;
            if (t >= q.tokens) break;
            if (t > 0 && (t & 31) == 0)
                token_scalars(q, b, h, bias, Ah, t, lane, lane_dtv, lane_dA);
            const float dtv = __shfl_sync(0xffffffffu, lane_dtv, t & 31);
            const float dA = __shfl_sync(0xffffffffu, lane_dA, t & 31);
            float2 b2[NC / 2], c2[NC / 2];
            widen_pairs<NC>(ring[k].b, b2);
            widen_pairs<NC>(ring[k].c, c2);
            const float2 dA2 = make_float2(dA, dA);
            const float xl = widen_bf16(ring[k].x);
            if (t + PD < q.tokens) load_token<NC, VEC>(Bn, Cn, xn, x_live, ring[k]);
            Bn += q.B_t;
            Cn += q.C_t;
            xn += q.x_t;
            const float kl = dtv * xl;  // lane r < RPW: dt * x of row r
            float part[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                part[r] = update_pairs<NC>(w[r], dA2, __shfl_sync(0xffffffffu, kl, r), b2, c2);
            if (q.inter) {
                ST *irow = static_cast<ST *>(q.inter) + b * q.in_b + t * q.in_t + h * q.in_h +
                           row0 * q.in_p + lo;
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    float tmp[NC];
#pragma unroll
                    for (int i = 0; i < NC / 2; ++i) {
                        tmp[2 * i] = w[r][i].x;
                        tmp[2 * i + 1] = w[r][i].y;
                    }
                    if (row0 + r < p.headdim) store_cols<NC, ST>(irow + r * q.in_p, tmp);
                }
            }
            const float total = reduce_rows<RPW>(part, lane);
            const int rl = row_of_lane<RPW>(lane);
            const float xr = __shfl_sync(0xffffffffu, xl, rl);
            if (writes_row<RPW>(lane) && row0 + rl < p.headdim)
                p.out[b * p.out_b + t * q.out_t + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) v[r][2 * i] = w[r][i].x, v[r][2 * i + 1] = w[r][i].y;
}

// 16 rows per warp hold 64 state values per lane: those CTAs are limited to 4 warps so the
// compiler may use up to 255 registers without spilling.
template <int RPW>
constexpr int tokens_max_threads() {
    return RPW >= 16 ? 128 : 32 * kMaxWarpsPerCta;
}

// Registers per thread: what the largest CTA allows (tokens_max_threads), except for the 8-row
// kernels up to dstate 128 (the table's shape), held to 96 so 20 warps fit on an SM; with a
// ring of 2 they need no spill at that cap (see kTokenPrefetch).
template <int RPW, int NC>
constexpr int tokens_max_regs() {
    return RPW == 8 && NC <= 4 ? 96 : (RPW >= 16 ? 255 : 65536 / tokens_max_threads<RPW>());
}

template <int RPW, int NC, typename ST, bool kIdx64, int PD>
__global__ void __maxnreg__((tokens_max_regs<RPW, NC>()))
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

        if (q.bc_vec)
            token_loop<RPW, NC, ST, true, PD>(q, v, b, h, row0, lane);
        else
            token_loop<RPW, NC, ST, false, PD>(q, v, b, h, row0, lane);
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            if (row0 + r < p.headdim) store_cols<NC, ST>(srow + r * p.st_row, v[r]);
    }
    pdl_trigger();  // this CTA's stores are issued: a dependent launch may start its CTAs
}

template <int RPW, int NC, typename ST, bool kIdx64, int PD>
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
    return cudaLaunchKernelEx(&cfg, ssu_tokens_kernel<RPW, NC, ST, kIdx64, PD>, q);
}

template <int NC, typename ST, bool kIdx64, int PD>
cudaError_t launch_tokens_t(const TokenParams &q, int rpw, int wpc, dim3 grid, bool pdl,
                            cudaStream_t st) {
    const dim3 block(32 * wpc);
    switch (rpw) {
        case 1: return launch_tokens_one<1, NC, ST, kIdx64, PD>(q, grid, block, pdl, st);
        case 2: return launch_tokens_one<2, NC, ST, kIdx64, PD>(q, grid, block, pdl, st);
        case 4: return launch_tokens_one<4, NC, ST, kIdx64, PD>(q, grid, block, pdl, st);
        case 8: return launch_tokens_one<8, NC, ST, kIdx64, PD>(q, grid, block, pdl, st);
        case 16:
            if constexpr (NC <= 4)
                return static_cast<int>(block.x) <= tokens_max_threads<16>()
                           ? launch_tokens_one<16, NC, ST, kIdx64, PD>(q, grid, block, pdl, st)
                           : cudaErrorInvalidValue;
            else
                return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

// Launches the multi-token kernel with a prefetch ring of PD tokens for dstate = 32 * nc, a
// bf16 or fp32 state, int64 or int32 indices.
template <int PD>
cudaError_t launch_tokens_depth(const TokenParams &q, int nc, bool bf16, bool i64, int rpw,
                                int wpc, dim3 grid, bool pdl, cudaStream_t st) {
#define SSU_TOK_T(NC_, ST_, I64_) launch_tokens_t<NC_, ST_, I64_, PD>(q, rpw, wpc, grid, pdl, st)
#define SSU_TOK_NC(NC_)                                                                 \
    if (nc == NC_) {                                                                    \
        if (bf16)                                                                       \
            return i64 ? SSU_TOK_T(NC_, __nv_bfloat16, true)                            \
                       : SSU_TOK_T(NC_, __nv_bfloat16, false);                          \
        return i64 ? SSU_TOK_T(NC_, float, true) : SSU_TOK_T(NC_, float, false);        \
    }
    SSU_TOK_NC(2)
    SSU_TOK_NC(4)
    SSU_TOK_NC(8)
#undef SSU_TOK_NC
#undef SSU_TOK_T
    return cudaErrorInvalidValue;
}

}  // namespace
