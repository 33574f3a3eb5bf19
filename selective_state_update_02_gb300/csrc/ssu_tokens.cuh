// Multi-token decode-step kernel for GB300 (sm_103a), instantiated by ssu_tokens.cu (which
// also holds the C entry point).
//
// The step: T consecutive tokens of every request in one call (the verification step of
// multi-token speculation, vLLM PR #48110, Test Plan).  Token t applies the single-token update
// to the state token t - 1 left; the state is loaded once, kept in registers (fp32) across the
// T tokens, and stored once.  Element mapping (RowGeo), update order and readout tree are the
// single-step kernel's, so T = 1 reproduces ssu_update bit for bit.
//
// Grid as the single-step kernel's: one CTA per (slab of rows, head, request), each warp RPW
// rows.  A warp issues its state loads, then the loads of its first tokens' inputs (held as raw
// bits in a register ring, PD tokens ahead) and its tokens' dt, so all of them are in flight
// together; it computes every token's dt and dA once per warp (lane j for token j, handed out
// by shuffles).  (A persistent variant, each warp streaming its next tiles' state into shared
// memory with cp.async while computing the current one, measured 1.5-1.8x slower: the first
// tokens' inputs of every tile were then waited for with nothing else in flight.)

#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ssu_device.cuh"

namespace {

struct TokenParams {
    SsuParams p;                       // p.slabs tiles per (request, head), p.rows_per_cta = RPW
    void *inter;                       // optional intermediate states (state dtype), may be null
    long long x_t, out_t, dt_t, B_t, C_t;
    long long in_b, in_t, in_h, in_p;  // intermediate strides; dstate stride is 1
    int tokens;
    int bc_vec;  // B and C rows can be read as whole column groups (aligned vectors)
};

// update_lane (ssu_device.cuh) on the lane's NC values of one row held as fp32 pairs (column
// 2i in .x, 2i+1 in .y): the same packed instructions and the same readout order, so the same
// values bit for bit.  Holding the state and B/C as pairs for the whole token loop saves the
// moves that form pairs out of scalar registers (measured 1-2 % faster at T >= 3).
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
// issued as soon as token t's inputs have been widened.  Two where a lane holds 4 columns of a
// row; one at 8 columns (dstate 256, a bf16 state), where a ring of two spills at 128
// registers (ptxas, CUDA 13.0).
template <int N, typename ST>
constexpr int token_prefetch() {
    return RowGeo<N, ST>::NC <= 4 ? 2 : 1;
}

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

// The lane's NC columns starting at `p` (its first column) as pair words.  VEC: one 8- or
// 16-byte load per column group (the host checked the alignment); otherwise two 2-byte loads
// per pair.
template <class G, bool VEC>
__device__ __forceinline__ void load_pairs(const unsigned short *p, unsigned (&w)[G::NC / 2]) {
    if constexpr (VEC) {
#pragma unroll
        for (int v = 0; v < G::VPR; ++v) {
            if constexpr (G::kEPV == 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(p + v * G::kVecStride);
                w[4 * v] = u.x, w[4 * v + 1] = u.y, w[4 * v + 2] = u.z, w[4 * v + 3] = u.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2 *>(p + v * G::kVecStride);
                w[2 * v] = u.x, w[2 * v + 1] = u.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < G::NC / 2; ++i) {
            const int e = 2 * i;
            const unsigned short *q = p + (e / G::kEPV) * G::kVecStride + e % G::kEPV;
            w[i] = static_cast<unsigned>(q[0]) | (static_cast<unsigned>(q[1]) << 16);
        }
    }
}

// One token's inputs into a ring slot: `B` and `C` point at the lane's first column of the
// token's rows, `x` at the lane's x element (read only where `x_live`: lanes r < RPW whose row
// exists).
template <class G, bool VEC>
__device__ __forceinline__ void load_token(const unsigned short *B, const unsigned short *C,
                                           const unsigned short *x, bool x_live,
                                           TokenBits<G::NC> &in) {
    load_pairs<G, VEC>(B, in.b);
    load_pairs<G, VEC>(C, in.c);
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

// The T-token loop of one warp over its tile (S vector rows held in w as fp32 pairs).  The
// per-token inputs are read through pointers built once per tile and advanced by one token
// stride per token; the outputs' addresses are formed per token (carrying output pointers
// through the loop as well measured 5-10 % slower once the ring refills).
template <int RPW, int N, typename ST, bool VEC, int PD>
__device__ __forceinline__ void token_loop(
    const TokenParams &q, float2 (&w)[RPW / RowGeo<N, ST>::RPI][RowGeo<N, ST>::NC / 2],
    long long b, int h, int row0, int lane) {
    using G = RowGeo<N, ST>;
    constexpr int S = RPW / G::RPI, NC = G::NC, RPI = G::RPI;
    const SsuParams &p = q.p;
    const int sub = sub_of<G>(lane);
    const float bias = p.dt_bias[h * p.bias_h];
    const float Ah = p.A[h * p.A_h];
    const float Dh = p.D[h * p.D_h];
    const int g = group_of(h, p.group_magic);
    const int c0 = col0_of<G>(lane);
    const unsigned short *Bn = reinterpret_cast<const unsigned short *>(p.B) + b * p.B_b +
                               g * p.B_g + c0;
    const unsigned short *Cn = reinterpret_cast<const unsigned short *>(p.C) + b * p.C_b +
                               g * p.C_g + c0;
    const bool x_live = lane < RPW && row0 + lane < p.headdim;
    const unsigned short *xn = reinterpret_cast<const unsigned short *>(p.x) + b * p.x_b +
                               h * p.x_h + row0 + (x_live ? lane : 0);
    // A ring of the next PD tokens' inputs, unrolled so every slot is a fixed register.
    TokenBits<NC> ring[PD];
#pragma unroll
    for (int k = 0; k < PD; ++k)
        if (k < q.tokens)
            load_token<G, VEC>(Bn + k * q.B_t, Cn + k * q.C_t, xn + k * q.x_t, x_live, ring[k]);
    Bn += PD * q.B_t;  // now token PD's
    Cn += PD * q.C_t;
    xn += PD * q.x_t;
    float lane_dtv, lane_dA;
    token_scalars(q, b, h, bias, Ah, 0, lane, lane_dtv, lane_dA);
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
            if (t + PD < q.tokens) load_token<G, VEC>(Bn, Cn, xn, x_live, ring[k]);
            Bn += q.B_t;
            Cn += q.C_t;
            xn += q.x_t;
            const float kl = dtv * xl;  // lane r < RPW: dt * x of row r
            float part[S];
#pragma unroll
            for (int r = 0; r < S; ++r)
                part[r] = update_pairs<NC>(w[r], dA2, __shfl_sync(0xffffffffu, kl, r * RPI + sub),
                                           b2, c2);
            if (q.inter) {
                ST *irow = static_cast<ST *>(q.inter) + b * q.in_b + t * q.in_t + h * q.in_h +
                           (row0 + sub) * q.in_p + c0;
                const long long islot = RPI * q.in_p;
#pragma unroll
                for (int r = 0; r < S; ++r) {
                    float tmp[NC];
#pragma unroll
                    for (int i = 0; i < NC / 2; ++i) tmp[2 * i] = w[r][i].x, tmp[2 * i + 1] = w[r][i].y;
                    RawRow<G> o;
                    f32_to_raw<G, ST>(tmp, o);
                    if (row0 + sub + r * RPI < p.headdim) store_raw<G, ST>(irow + r * islot, o);
                }
            }
            const float total = reduce_rows<S, G::L>(part, lane);
            const int rl = slot_of_lane<S, G::L>(lane) * RPI + sub;  // row within the tile
            const float xr = __shfl_sync(0xffffffffu, xl, rl);
            if (writes_row<S, G::L>(lane) && row0 + rl < p.headdim)
                p.out[b * p.out_b + t * q.out_t + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
        }
    }
}

// Registers per thread: 96 for a tile of at most 32 fp32 state values per lane, so 20 warps
// fit on an SM (5 per sub-partition's register file): fp32 dstate 128 at 8 rows spills 8
// bytes there (ptxas, CUDA 13.0) and still ran faster than at 104 registers without a spill
// (T = 3 / 4 / 8: 26.6 / 29.4 / 40.2 against 27.5 / 31.3 / 43.4 us).  Larger tiles (a bf16
// state's 64 values) take 128, where they need no spill.
template <int RPW, int N, typename ST>
constexpr int tokens_max_regs() {
    using G = RowGeo<N, ST>;
    return (RPW / G::RPI) * G::NC <= 32 ? 96 : 128;
}

template <int RPW, int N, typename ST, bool kIdx64, int PD>
__global__ void __maxnreg__((tokens_max_regs<RPW, N, ST>()))
    ssu_tokens_kernel(const __grid_constant__ TokenParams q) {
    using G = RowGeo<N, ST>;
    constexpr int S = RPW / G::RPI, NC = G::NC, RPI = G::RPI;
    pdl_wait();
    const SsuParams &p = q.p;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int slab = blockIdx.x;
    const int h = blockIdx.y;
    const int sub = sub_of<G>(lane);
    for (long long b = blockIdx.z; b < p.batch; b += gridDim.z) {
        const long long s = load_slot<kIdx64>(p, b);
        if (s < 0 || s >= p.pool_size) {
            if (h == 0 && slab == 0 && threadIdx.x == 0) record_skip(p, b);
            continue;
        }
        const int row0 = slab * p.rows_per_cta + warp * RPW;
        const int lrow = row0 + sub;
        ST *srow = static_cast<ST *>(p.state) + s * p.st_pool + h * p.st_head +
                   lrow * p.st_row + col0_of<G>(lane);
        RawRow<G> raw[S];
#pragma unroll
        for (int r = 0; r < S; ++r) {
            if (lrow + r * RPI < p.headdim) {
                load_raw<G, ST>(srow + r * RPI * p.st_row, raw[r]);
            } else {
#pragma unroll
                for (int v = 0; v < G::VPR; ++v) raw[r].w[v] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float2 w[S][NC / 2];
#pragma unroll
        for (int r = 0; r < S; ++r) {
            float f[NC];
            raw_to_f32<G, ST>(raw[r], f);
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) w[r][i] = make_float2(f[2 * i], f[2 * i + 1]);
        }
        if (q.bc_vec)
            token_loop<RPW, N, ST, true, PD>(q, w, b, h, row0, lane);
        else
            token_loop<RPW, N, ST, false, PD>(q, w, b, h, row0, lane);
#pragma unroll
        for (int r = 0; r < S; ++r) {
            if (lrow + r * RPI < p.headdim) {
                float f[NC];
#pragma unroll
                for (int i = 0; i < NC / 2; ++i) f[2 * i] = w[r][i].x, f[2 * i + 1] = w[r][i].y;
                RawRow<G> o;
                f32_to_raw<G, ST>(f, o);
                store_raw<G, ST>(srow + r * RPI * p.st_row, o);
            }
        }
    }
    pdl_trigger();  // this CTA's stores are issued: a dependent launch may start its CTAs
}

template <int RPW, int N, typename ST, bool kIdx64, int PD>
cudaError_t launch_tokens_one(const TokenParams &q, dim3 grid, int warps, bool pdl,
                              cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * warps);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ssu_tokens_kernel<RPW, N, ST, kIdx64, PD>, q);
}

}  // namespace
