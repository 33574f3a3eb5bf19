// VEC kernel of the decode step: one CTA per (slab of rows, head, request).  Each warp holds
// RPW rows of the state in registers as whole 16-byte vectors (all loads issued before any
// use), updates them, stores them back in place with streaming stores and writes the readout.
// Templated on the rows per warp, dstate, the state element type (fp32 or bf16, computed in
// fp32 either way) and the index type; the lane geometry of a row is RowGeo (ssu_device.cuh).
#pragma once

#include "ssu_device.cuh"

namespace {

// Per-instantiation forms of the per-row work, each chosen from a same-box A/B at batch 128
// (and 8 / 512 for fp32 at dstate 128), since the compiler's schedules differ:
//  * kShuffleK: lane r < RPW loads x of row r and forms dt * x there; the other lanes get the
//    product by a shuffle (instead of every lane loading every row's x and multiplying).  On
//    wherever one instruction covers several rows (the lanes of one instruction need
//    different rows' products), for a bf16 state, and for fp32 with 8 rows per warp at dstate
//    128; off for fp32 with 2 rows per warp (batch 8: 3.56 -> 3.91 us with it) and at dstate
//    256.
//  * kVectorBC: B and C read as whole column groups (8 or 16 bytes per lane) when aligned.  On
//    at dstate 256 (fp32 41.52 -> 41.14), for fp32 with 8 rows per warp at dstate 128 (22.99 ->
//    22.76 at batch 128, 81.03 -> 80.56 at 512) and wherever one instruction covers several
//    rows.
//  * kGroupMagic: the head's group from group_of (a multiply and a shift) instead of an integer
//    division.  On with 8 rows per warp for fp32 at dstate 128 (22.76 -> 22.65 at batch 128,
//    80.68 -> 80.53 at 512) and for bf16 at dstate 256 (24.67 -> 24.55); off for fp32 with 2
//    rows per warp (batch 8: 3.56 -> 3.95).
//  * kPacked: the state update in packed fp32x2 multiplies and fused multiply-adds (IEEE round
//    to nearest per element, the same values).  On for a bf16 state, for fp32 with 8 rows per
//    warp at dstate 128 (22.34 -> 22.27 at batch 128) and wherever one instruction covers
//    several rows; off for fp32 at dstate 256 (40.94 -> 42.30 with it: more registers, fewer
//    warps).
// Every combination gives the same values bit for bit.
template <int RPW, int N, typename ST>
struct VecForm {
    using G = RowGeo<N, ST>;
    static constexpr int S = RPW / G::RPI;  // vector instructions (slots) per warp
    static constexpr bool kMulti = G::RPI > 1;
    static constexpr bool kShuffleK = kMulti || sizeof(ST) == 2 || (N == 128 && RPW >= 8);
    static constexpr bool kVectorBC = kMulti || N == 256 || (N == 128 && RPW >= 8);
    static constexpr bool kGroupMagic = kMulti || (RPW >= 8 && G::NC * sizeof(ST) == 16);
    static constexpr bool kPacked = kMulti || sizeof(ST) == 2 || (N == 128 && RPW == 8);
    static_assert(RPW % G::RPI == 0 && S >= 1 && S <= G::L, "rows per warp for this dstate");
};

template <int RPW, int N, typename ST>
__device__ __forceinline__ float update_row(float (&v)[RowGeo<N, ST>::NC], float dA, float k,
                                            const float (&bb)[RowGeo<N, ST>::NC],
                                            const float (&cc)[RowGeo<N, ST>::NC]) {
    constexpr int NC = RowGeo<N, ST>::NC;
    if constexpr (VecForm<RPW, N, ST>::kPacked)
        return update_lane<NC>(v, dA, k, bb, cc);
    else
        return update_lane_scalar<NC>(v, dA, k, bb, cc);
}

// Registers per thread for an instantiation.  Under the launch bound of a 16-warp CTA alone
// the compiler takes far more than it needs for some (fp32 dstate 64 with 16 rows per warp:
// 118; bf16 with 8 vector rows: 103-108; dstate 256 with 4 vector rows: 115-117; fp32 dstate
// 128 with 16 rows: 128 and a spill), which costs resident warps; those are compiled as
// ssu_vec_kernel_capped, held to the smallest multiple of 8 at which ptxas (CUDA 13.0,
// sm_103a) keeps every variable in registers (fp32 dstate 128 at 8 rows: 74 -> 64, the 32
// warps per SM its timing rests on).  The others (128 here) keep the launch bound only: a
// register cap they do not need changed their schedules (fp32 dstate 128 with 2 rows per
// warp: 40 -> 44 registers under a cap of 64, batch 8 at 3.84 instead of 3.38 us).
template <int RPW, int N, typename ST>
constexpr int vec_max_regs() {
    using G = RowGeo<N, ST>;
    constexpr int S = RPW / G::RPI, V = S * G::VPR;  // 16-byte vectors of state per lane
    if constexpr (sizeof(ST) == 4) {
        if (V >= 16) return 104;            // fp32 dstate 128 at 16 rows, dstate 256 at 8
        if (V == 8) return G::VPR == 2 ? 72 : 64;
        return 128;
    }
    if (S >= 8) return 96;
    if (S == 4) return 72;
    return 128;
}

// The decode step of one CTA.  Grid: x = slab of rows, y = head, z = request (requests beyond
// gridDim.z loop), so the slot lookup at the head of the dependency chain needs no index
// arithmetic.
template <int RPW, int N, typename ST, bool kIdx64>
__device__ __forceinline__ void vec_step(const SsuParams &p) {
    using G = RowGeo<N, ST>;
    using F = VecForm<RPW, N, ST>;
    constexpr int S = F::S, NC = G::NC, RPI = G::RPI;
    pdl_wait();
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

        const int row0 = slab * p.rows_per_cta + warp * RPW;  // the warp's first row
        const int lrow = row0 + sub;                           // the lane's row in slot 0
        ST *srow = static_cast<ST *>(p.state) + s * p.st_pool + h * p.st_head +
                   lrow * p.st_row + col0_of<G>(lane);
        const long long slot_stride = RPI * p.st_row;

        // Issue every state load of this warp before anything that depends on other loads.
        RawRow<G> raw[S];
#pragma unroll
        for (int r = 0; r < S; ++r) {
            if (lrow + r * RPI < p.headdim) {
                load_raw<G, ST>(srow + r * slot_stride, raw[r]);
            } else {
#pragma unroll
                for (int q = 0; q < G::VPR; ++q) raw[r].w[q] = make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // Per-unit scalars, computed while the state loads are in flight.
        const float z =
            __bfloat162float(p.dt[b * p.dt_b + h * p.dt_h]) + p.dt_bias[h * p.bias_h];
        const float dtv = softplus_f32(z);
        const float dA = expf(dtv * p.A[h * p.A_h]);
        const float Dh = p.D[h * p.D_h];
        const int g = F::kGroupMagic ? group_of(h, p.group_magic) : h / p.heads_per_group;
        float bb[NC], cc[NC];
        const __nv_bfloat16 *Bw = p.B + b * p.B_b + g * p.B_g, *Cw = p.C + b * p.C_b + g * p.C_g;
        const bool bc_vec =
            F::kVectorBC &&
            ((reinterpret_cast<unsigned long long>(Bw) | reinterpret_cast<unsigned long long>(Cw)) &
             (2 * G::kEPV - 1)) == 0;
        // Two call sites with a constant flag each: one path with the flag as a run-time
        // argument measured 8 more registers (72 instead of 64 at 8 rows, fp32, dstate 128).
        if (bc_vec) {
            load_bc<G>(Bw + col0_of<G>(lane), true, bb);
            load_bc<G>(Cw + col0_of<G>(lane), true, cc);
        } else {
            load_bc<G>(Bw + col0_of<G>(lane), false, bb);
            load_bc<G>(Cw + col0_of<G>(lane), false, cc);
        }
        const __nv_bfloat16 *xp = p.x + b * p.x_b + h * p.x_h + row0;
        float part[S];
        if constexpr (F::kShuffleK) {
            const bool x_live = lane < RPW && row0 + lane < p.headdim;
            const float xl = x_live ? __bfloat162float(xp[lane]) : 0.f;
            const float kl = dtv * xl;  // lane r < RPW: dt * x of row r
#pragma unroll
            for (int r = 0; r < S; ++r) {
                float v[NC];
                raw_to_f32<G, ST>(raw[r], v);
                part[r] = update_row<RPW, N, ST>(v, dA, __shfl_sync(0xffffffffu, kl, r * RPI + sub),
                                                 bb, cc);
                if (lrow + r * RPI < p.headdim) {
                    RawRow<G> o;
                    f32_to_raw<G, ST>(v, o);
                    store_raw<G, ST>(srow + r * slot_stride, o);
                }
            }
            const float total = reduce_rows<S, G::L>(part, lane);
            const int rl = slot_of_lane<S, G::L>(lane) * RPI + sub;  // row within the warp
            const float xr = __shfl_sync(0xffffffffu, xl, rl);
            if (writes_row<S, G::L>(lane) && row0 + rl < p.headdim)
                p.out[b * p.out_b + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
        } else {
            static_assert(RPI == 1, "several rows per instruction need the shuffled dt * x");
#pragma unroll
            for (int r = 0; r < S; ++r) {
                const bool live = row0 + r < p.headdim;
                const float xr = live ? __bfloat162float(xp[r]) : 0.f;
                float v[NC];
                raw_to_f32<G, ST>(raw[r], v);
                part[r] = update_row<RPW, N, ST>(v, dA, dtv * xr, bb, cc);
                if (live) {
                    RawRow<G> o;
                    f32_to_raw<G, ST>(v, o);
                    store_raw<G, ST>(srow + r * slot_stride, o);
                }
            }
            const float total = reduce_rows<S, G::L>(part, lane);
            const int rl = slot_of_lane<S, G::L>(lane);
            if (writes_row<S, G::L>(lane) && row0 + rl < p.headdim) {
                const float xr = __bfloat162float(xp[rl]);
                p.out[b * p.out_b + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
            }
        }
    }
    pdl_trigger();  // this CTA's stores are issued: a dependent launch may start its CTAs
}

template <int RPW, int N, typename ST, bool kIdx64>
__global__ void __launch_bounds__(32 * kMaxWarpsPerCta)
    ssu_vec_kernel(const __grid_constant__ SsuParams p) {
    vec_step<RPW, N, ST, kIdx64>(p);
}

template <int RPW, int N, typename ST, bool kIdx64>
__global__ void __maxnreg__((vec_max_regs<RPW, N, ST>()))
    ssu_vec_kernel_capped(const __grid_constant__ SsuParams p) {
    vec_step<RPW, N, ST, kIdx64>(p);
}

// Launches one instantiation; with `pdl` the launch may begin before the previous kernel in
// the stream has finished (the kernel waits for it before touching memory).
template <int RPW, int N, typename ST, bool kIdx64>
cudaError_t launch_vec_one(const SsuParams &p, dim3 grid, dim3 block, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if constexpr (vec_max_regs<RPW, N, ST>() < 128)
        return cudaLaunchKernelEx(&cfg, ssu_vec_kernel_capped<RPW, N, ST, kIdx64>, p);
    else
        return cudaLaunchKernelEx(&cfg, ssu_vec_kernel<RPW, N, ST, kIdx64>, p);
}

// Rows per warp this build instantiates for a (dstate, state type): RPI x {1, 2, 4, 8}, and 16
// for an fp32 state of dstate 128.
template <int N, typename ST, bool kIdx64>
cudaError_t launch_vec_t(const SsuParams &p, int rpw, int wpc, dim3 grid, bool pdl,
                         cudaStream_t st) {
    constexpr int RPI = RowGeo<N, ST>::RPI;
    const dim3 block(32 * wpc);
    if (rpw == RPI) return launch_vec_one<RPI, N, ST, kIdx64>(p, grid, block, pdl, st);
    if (rpw == 2 * RPI) return launch_vec_one<2 * RPI, N, ST, kIdx64>(p, grid, block, pdl, st);
    if (rpw == 4 * RPI) return launch_vec_one<4 * RPI, N, ST, kIdx64>(p, grid, block, pdl, st);
    if (rpw == 8 * RPI) return launch_vec_one<8 * RPI, N, ST, kIdx64>(p, grid, block, pdl, st);
    if constexpr (N == 128 && sizeof(ST) == 4)
        if (rpw == 16) return launch_vec_one<16, N, ST, kIdx64>(p, grid, block, pdl, st);
    return cudaErrorInvalidValue;
}

// Launches the VEC kernel for dstate 64, 128 or 256, a bf16 or fp32 state, int64 or int32
// indices.
inline cudaError_t launch_vec(const SsuParams &p, int dstate, bool bf16, bool i64, int rpw,
                              int wpc, dim3 grid, bool pdl, cudaStream_t st) {
#define SSU_VEC_N(N_)                                                                      \
    if (dstate == N_) {                                                                    \
        if (bf16)                                                                          \
            return i64 ? launch_vec_t<N_, __nv_bfloat16, true>(p, rpw, wpc, grid, pdl, st) \
                       : launch_vec_t<N_, __nv_bfloat16, false>(p, rpw, wpc, grid, pdl, st); \
        return i64 ? launch_vec_t<N_, float, true>(p, rpw, wpc, grid, pdl, st)             \
                   : launch_vec_t<N_, float, false>(p, rpw, wpc, grid, pdl, st);           \
    }
    SSU_VEC_N(64)
    SSU_VEC_N(128)
    SSU_VEC_N(256)
#undef SSU_VEC_N
    return cudaErrorInvalidValue;
}

}  // namespace
