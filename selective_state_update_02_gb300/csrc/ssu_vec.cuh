// VEC kernel of the decode step: one CTA per (slab of rows, head, request).  Each warp holds
// RPW rows of the state in registers (all loads issued before any use), updates them, stores
// them back in place with streaming stores and writes the readout.  Templated on the rows per
// warp, the columns per lane (dstate = 32 * NC), the state element type (fp32 or bf16, computed
// in fp32 either way) and the index type.
#pragma once

#include "ssu_device.cuh"

namespace {

// The lane's NC columns of B (or C) widened to fp32, read as whole 4- or 8-byte column groups.
// Only for a warp whose first column address is aligned to that width (every lane then is).
template <int NC>
__device__ __forceinline__ void load_bc_vec(const __nv_bfloat16 *p, float (&o)[NC]) {
    unsigned w[NC / 2];
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
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Per-instantiation forms of the per-row work, each chosen from a same-box A/B at batch 128
// (and 8 / 512 for fp32 at dstate 128), since the compiler's schedules differ:
//  * kShuffleK: lane r < RPW loads x of row r and forms dt * x there; the other lanes get the
//    product by a shuffle (instead of every lane loading every row's x and multiplying).  On
//    for a bf16 state (dstate 128: 14.88 -> 13.78 us; 64: 11.91 -> 10.72) and for fp32 with 8
//    rows per warp at dstate 128; off for fp32 at dstate 64 (13.26 -> 13.70) and with 2 rows
//    per warp (batch 8: 3.56 -> 3.91).
//  * kVectorBC: B and C read as 4- or 8-byte column groups when aligned.  On at dstate 256
//    (bf16 26.51 -> 24.63; fp32 41.52 -> 41.14) and for fp32 with 8 rows per warp at dstate
//    128 (both on: 22.99 -> 22.76 at batch 128, 81.03 -> 80.56 at 512); off at dstate 64
//    (fp32 13.26 -> 14.61).
//  * kGroupMagic: the head's group from group_of (a multiply and a shift) instead of an integer
//    division.  On with 8 rows per warp where a lane's part of a row is one 16-byte vector
//    (fp32 at dstate 128: 22.76 -> 22.65 at batch 128, 80.68 -> 80.53 at 512; bf16 at dstate
//    256: 24.67 -> 24.55); off elsewhere (fp32 batch 8: 3.56 -> 3.95; bf16 dstate 128: 13.84
//    -> 15.43; dstate 64 fp32 13.29 -> 13.74, bf16 10.74 -> 11.12; fp32 dstate 256 unchanged).
//  * kPacked: the state update in packed fp32x2 multiplies and fused multiply-adds (IEEE round
//    to nearest per element, the same values).  On for a bf16 state (dstate 128 / 256 / 64:
//    13.50 -> 13.42, 24.22 -> 24.07, 10.59 -> 10.47 us at batch 128) and for fp32 with 8 rows
//    per warp at dstate 128 (22.34 -> 22.27 at batch 128, 80.17 -> 80.09 at 512); off for fp32
//    at dstate 64 and 256 (13.00 -> 13.56, 40.94 -> 42.30: more registers, fewer warps).
// Every combination gives the same values bit for bit.
template <int RPW, int NC, typename ST>
struct VecForm {
    static constexpr bool kShuffleK = sizeof(ST) == 2 || (NC == 4 && RPW >= 8);
    static constexpr bool kVectorBC = NC == 8 || (NC == 4 && sizeof(ST) == 4 && RPW >= 8);
    static constexpr bool kGroupMagic = RPW >= 8 && NC * sizeof(ST) == 16;
    static constexpr bool kPacked = sizeof(ST) == 2 || (NC == 4 && RPW == 8);
};

// update_lane (ssu_device.cuh) with the state update in packed fp32x2 instructions; the
// readout chain stays scalar, over the columns in the same order.
template <int NC>
__device__ __forceinline__ float update_lane_packed(float (&v)[NC], float dA, float k,
                                                    const float (&bb)[NC],
                                                    const float (&cc)[NC]) {
    const float2 k2 = make_float2(k, k), dA2 = make_float2(dA, dA);
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) {
        const float2 w = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), dA2,
                                    __fmul2_rn(k2, make_float2(bb[2 * i], bb[2 * i + 1])));
        v[2 * i] = w.x;
        v[2 * i + 1] = w.y;
    }
    float part = v[0] * cc[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) part = fmaf(v[j], cc[j], part);
    return part;
}

template <int RPW, int NC, typename ST>
__device__ __forceinline__ float update_row(float (&v)[NC], float dA, float k,
                                            const float (&bb)[NC], const float (&cc)[NC]) {
    if constexpr (VecForm<RPW, NC, ST>::kPacked)
        return update_lane_packed<NC>(v, dA, k, bb, cc);
    else
        return update_lane<NC>(v, dA, k, bb, cc);
}

// Grid: x = slab of rows, y = head, z = request (requests beyond gridDim.z loop), so the
// slot lookup at the head of the dependency chain needs no index arithmetic.
template <int RPW, int NC, typename ST, bool kIdx64>
__global__ void __launch_bounds__(32 * kMaxWarpsPerCta)
    ssu_vec_kernel(const __grid_constant__ SsuParams p) {
    pdl_wait();
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

        // Issue every state load of this warp before anything that depends on other loads.
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

        // Per-unit scalars, computed while the state loads are in flight.
        const float z =
            __bfloat162float(p.dt[b * p.dt_b + h * p.dt_h]) + p.dt_bias[h * p.bias_h];
        const float dtv = softplus_f32(z);
        const float dA = expf(dtv * p.A[h * p.A_h]);
        const float Dh = p.D[h * p.D_h];
        const int g = VecForm<RPW, NC, ST>::kGroupMagic ? group_of(h, p.group_magic)
                                                        : h / p.heads_per_group;
        float bb[NC], cc[NC];
        const __nv_bfloat16 *Bw = p.B + b * p.B_b + g * p.B_g, *Cw = p.C + b * p.C_b + g * p.C_g;
        if (VecForm<RPW, NC, ST>::kVectorBC &&
            ((reinterpret_cast<unsigned long long>(Bw) | reinterpret_cast<unsigned long long>(Cw)) &
             (NC == 2 ? 3u : 7u)) == 0) {
            load_bc_vec<NC>(Bw + lane_offset<NC>(lane), bb);
            load_bc_vec<NC>(Cw + lane_offset<NC>(lane), cc);
        } else {
            load_bc<NC>(Bw + lane_offset<NC>(lane), bb);
            load_bc<NC>(Cw + lane_offset<NC>(lane), cc);
        }
        const __nv_bfloat16 *xp = p.x + b * p.x_b + h * p.x_h + row0;
        float part[RPW];
        if constexpr (VecForm<RPW, NC, ST>::kShuffleK) {
            const bool x_live = lane < RPW && row0 + lane < p.headdim;
            const float xl = x_live ? __bfloat162float(xp[lane]) : 0.f;
            const float kl = dtv * xl;  // lane r < RPW: dt * x of row r
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                part[r] = update_row<RPW, NC, ST>(v[r], dA, __shfl_sync(0xffffffffu, kl, r), bb, cc);
                if (row0 + r < p.headdim) store_cols<NC, ST>(srow + r * p.st_row, v[r]);
            }
            const float total = reduce_rows<RPW>(part, lane);
            const int rl = row_of_lane<RPW>(lane);
            const float xr = __shfl_sync(0xffffffffu, xl, rl);
            if (writes_row<RPW>(lane) && row0 + rl < p.headdim)
                p.out[b * p.out_b + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
        } else {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const bool live = row0 + r < p.headdim;
                const float xr = live ? __bfloat162float(xp[r]) : 0.f;
                part[r] = update_row<RPW, NC, ST>(v[r], dA, dtv * xr, bb, cc);
                if (live) store_cols<NC, ST>(srow + r * p.st_row, v[r]);
            }
            const float total = reduce_rows<RPW>(part, lane);
            const int rl = row_of_lane<RPW>(lane);
            if (writes_row<RPW>(lane) && row0 + rl < p.headdim) {
                const float xr = __bfloat162float(xp[rl]);
                p.out[b * p.out_b + h * p.out_h + row0 + rl] =
                    __float2bfloat16_rn(fmaf(Dh, xr, total));
            }
        }
    }
    pdl_trigger();  // this CTA's stores are issued: a dependent launch may start its CTAs
}

// Launches one instantiation; with `pdl` the launch may begin before the previous kernel in
// the stream has finished (the kernel waits for it before touching memory).
template <int RPW, int NC, typename ST, bool kIdx64>
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
    return cudaLaunchKernelEx(&cfg, ssu_vec_kernel<RPW, NC, ST, kIdx64>, p);
}

template <int NC, typename ST, bool kIdx64>
cudaError_t launch_vec_t(const SsuParams &p, int rpw, int wpc, dim3 grid, bool pdl,
                         cudaStream_t st) {
    const dim3 block(32 * wpc);
    switch (rpw) {
        case 1: return launch_vec_one<1, NC, ST, kIdx64>(p, grid, block, pdl, st);
        case 2: return launch_vec_one<2, NC, ST, kIdx64>(p, grid, block, pdl, st);
        case 4: return launch_vec_one<4, NC, ST, kIdx64>(p, grid, block, pdl, st);
        case 8: return launch_vec_one<8, NC, ST, kIdx64>(p, grid, block, pdl, st);
        case 16:
            if constexpr (NC == 4 && sizeof(ST) == 4)
                return launch_vec_one<16, NC, ST, kIdx64>(p, grid, block, pdl, st);
            else
                return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

// Launches the VEC kernel for dstate = 32 * nc, a bf16 or fp32 state, int64 or int32 indices.
inline cudaError_t launch_vec(const SsuParams &p, int nc, bool bf16, bool i64, int rpw, int wpc,
                              dim3 grid, bool pdl, cudaStream_t st) {
#define SSU_VEC_NC(NC_)                                                                     \
    if (nc == NC_) {                                                                        \
        if (bf16)                                                                           \
            return i64 ? launch_vec_t<NC_, __nv_bfloat16, true>(p, rpw, wpc, grid, pdl, st) \
                       : launch_vec_t<NC_, __nv_bfloat16, false>(p, rpw, wpc, grid, pdl, st); \
        return i64 ? launch_vec_t<NC_, float, true>(p, rpw, wpc, grid, pdl, st)             \
                   : launch_vec_t<NC_, float, false>(p, rpw, wpc, grid, pdl, st);           \
    }
    SSU_VEC_NC(2)
    SSU_VEC_NC(4)
    SSU_VEC_NC(8)
#undef SSU_VEC_NC
    return cudaErrorInvalidValue;
}

}  // namespace
