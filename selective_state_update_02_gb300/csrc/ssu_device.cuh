// Device-side pieces shared by the decode-step kernels: launch constants, the parameter block,
// the per-element arithmetic, the readout reduction, slot lookup and programmatic dependent
// launch.  Included by each kernel translation unit (internal linkage per unit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kMaxWarpsPerCta = 16;

// Everything one launch needs, passed by value in the kernel parameter space.
struct SsuParams {
    void *state;  // fp32 or bf16 elements (the kernel's template parameter says which)
    const void *idx;
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *dt;
    const float *dt_bias;
    const float *A;
    const __nv_bfloat16 *B;
    const __nv_bfloat16 *C;
    const float *D;
    __nv_bfloat16 *out;
    long long st_pool, st_head, st_row;  // state strides (elements); dstate stride is 1
    long long x_b, x_h, out_b, out_h, dt_b, dt_h;
    long long B_b, B_g, C_b, C_g;
    long long bias_h, D_h, A_h, idx_s;
    long long pool_size;
    long long batch;
    int nheads, headdim, heads_per_group;
    unsigned long long group_magic;  // group_magic(heads_per_group): see group_of
    int slabs;         // tiles per (request, head) unit
    int rows_per_cta;  // rows per tile
    unsigned *err;     // [0] skipped requests, [1] smallest skipped request
};

// Group of head h, floor(h / d) for d = heads per group, without an integer division (the
// division by a value known only at run time expands into a long instruction sequence).  With
// m = floor(2^32 / d) + 1 = 2^32 / d + e, 0 < e <= 1:  h m / 2^32 = h / d + h e / 2^32, and
// for h, d < 2^16 the second term is below 2^-16 < 1 / d, so it cannot carry h / d past the
// next integer: floor(h m / 2^32) = floor(h / d).  Heads are limited to 65535.
__host__ __device__ inline unsigned long long group_magic(unsigned d) {
    return (1ull << 32) / d + 1;
}

__host__ __device__ __forceinline__ int group_of(int h, unsigned long long m) {
    return static_cast<int>((static_cast<unsigned long long>(h) * m) >> 32);
}

__device__ __forceinline__ float softplus_f32(float z) {
    // log(1 + e^z); above 20 the correction is below fp32 resolution of z.
    return z > 20.0f ? z : log1pf(expf(z));
}

// ---------------------------------------------------------------------------------------
// Lane geometry of a state row.  A row of dstate N elements of type ST (N * sizeof(ST) bytes)
// is read with 16-byte vectors.  A row of 512 bytes or more spreads over all 32 lanes, each
// lane holding VPR = bytes / 512 vectors (column groups L * EPV apart).  A shorter row (256 or
// 128 bytes) spreads over L = 16 or 8 lanes, so one warp-wide vector instruction covers
// RPI = 32 / L consecutive rows: lane l works on row-in-instruction l / L, column group l % L.
// Every warp-wide load or store thus moves 512 contiguous bytes of a contiguous state, and the
// per-warp work (slot lookup, scalars, addresses, the readout tree's shuffles) is spread over
// 512 bytes per instruction whatever the row size.
//
//   dstate, state   row bytes   L    RPI   columns per lane (NC)
//   64, fp32        256         16   2     4
//   128, fp32       512         32   1     4
//   256, fp32       1024        32   1     8  (4 + 4, 128 apart)
//   64, bf16        128         8    4     8
//   128, bf16       256         16   2     8
//   256, bf16       512         32   1     8
//
// A lane's e-th value is column (e / EPV) * L * EPV + (l % L) * EPV + e % EPV.  A "slot" is
// what one vector instruction of a warp covers: RPI rows.  The readout of a row sums the
// lane's NC products in order e = 0, 1, ... and then the L lanes of the row by the xor tree
// L/2, ..., 2, 1 (reduce_rows); every kernel and launch shape uses that order, so all give
// the same bits.
template <int N, typename ST>
struct RowGeo {
    static constexpr int kEPV = 16 / static_cast<int>(sizeof(ST));  // elements per vector
    static constexpr int kRowBytes = N * static_cast<int>(sizeof(ST));
    static constexpr int L = kRowBytes >= 512 ? 32 : kRowBytes / 16;
    static constexpr int RPI = 32 / L;
    static constexpr int VPR = kRowBytes >= 512 ? kRowBytes / 512 : 1;
    static constexpr int NC = VPR * kEPV;
    static constexpr int kVecStride = L * kEPV;  // columns between a lane's vectors
    static_assert(kRowBytes >= 128 && kRowBytes <= 1024, "dstate 64, 128 or 256");
};

// Offset (elements) of the lane's first column within its row.
template <class G>
__device__ __forceinline__ int col0_of(int lane) {
    return G::L == 32 ? lane * G::kEPV : (lane & (G::L - 1)) * G::kEPV;
}

// Row of the lane within one vector instruction (0 .. RPI - 1).
template <class G>
__device__ __forceinline__ int sub_of(int lane) {
    return G::RPI == 1 ? 0 : lane / G::L;
}

// A lane's share of one row as loaded: VPR 16-byte vectors.
template <class G>
struct RawRow {
    uint4 w[G::VPR];
};

// Streaming (evict-first) load of the lane's vectors of a row; `p` points at its first column.
template <class G, typename ST>
__device__ __forceinline__ void load_raw(const ST *p, RawRow<G> &r) {
#pragma unroll
    for (int v = 0; v < G::VPR; ++v)
        r.w[v] = __ldcs(reinterpret_cast<const uint4 *>(p + v * G::kVecStride));
}

template <class G, typename ST>
__device__ __forceinline__ void store_raw(ST *p, const RawRow<G> &r) {
#pragma unroll
    for (int v = 0; v < G::VPR; ++v)
        __stcs(reinterpret_cast<uint4 *>(p + v * G::kVecStride), r.w[v]);
}

__device__ __forceinline__ unsigned f2_to_bf2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // round to nearest even
    return *reinterpret_cast<const unsigned *>(&h);
}

// The lane's NC values of a row as fp32 (bf16 widens exactly: it is the top half of an fp32).
template <class G, typename ST>
__device__ __forceinline__ void raw_to_f32(const RawRow<G> &r, float (&v)[G::NC]) {
#pragma unroll
    for (int q = 0; q < G::VPR; ++q) {
        const unsigned w[4] = {r.w[q].x, r.w[q].y, r.w[q].z, r.w[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (sizeof(ST) == 4) {
                v[4 * q + i] = __uint_as_float(w[i]);
            } else {
                v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
                v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        }
    }
}

// The values back in the state's format (a bf16 state rounds to nearest even).
template <class G, typename ST>
__device__ __forceinline__ void f32_to_raw(const float (&v)[G::NC], RawRow<G> &r) {
#pragma unroll
    for (int q = 0; q < G::VPR; ++q) {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (sizeof(ST) == 4)
                w[i] = __float_as_uint(v[4 * q + i]);
            else
                w[i] = f2_to_bf2(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        }
        r.w[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The lane's NC columns of B (or C) widened to fp32; `p` points at its first column.  With
// `vec` (the warp found the row's address aligned to a whole column group: 2 * EPV bytes), one
// load per group; otherwise element by element.
template <class G>
__device__ __forceinline__ void load_bc(const __nv_bfloat16 *p, bool vec, float (&o)[G::NC]) {
    const unsigned short *q = reinterpret_cast<const unsigned short *>(p);
    if (vec) {
#pragma unroll
        for (int v = 0; v < G::VPR; ++v) {
            unsigned w[G::kEPV / 2];
            if constexpr (G::kEPV == 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(q + v * G::kVecStride);
                w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2 *>(q + v * G::kVecStride);
                w[0] = u.x, w[1] = u.y;
            }
#pragma unroll
            for (int i = 0; i < G::kEPV / 2; ++i) {
                o[v * G::kEPV + 2 * i] = __uint_as_float(w[i] << 16);
                o[v * G::kEPV + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < G::NC; ++e)
            o[e] = __uint_as_float(
                static_cast<unsigned>(q[(e / G::kEPV) * G::kVecStride + e % G::kEPV]) << 16);
    }
}

// The update of the lane's NC values of one row, S' = S dA + k B (k = dt x of the row), in
// packed fp32x2 instructions (IEEE round to nearest per element: the values of fmaf(S, dA,
// k * B)); returns the lane's part of the readout, its products S' C summed in order.
template <int NC>
__device__ __forceinline__ float update_lane(float (&v)[NC], float dA, float k,
                                             const float (&bb)[NC], const float (&cc)[NC]) {
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

// The same values by scalar instructions (fmaf(S, dA, k * B) per element).
template <int NC>
__device__ __forceinline__ float update_lane_scalar(float (&v)[NC], float dA, float k,
                                                    const float (&bb)[NC],
                                                    const float (&cc)[NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) v[j] = fmaf(v[j], dA, k * bb[j]);
    float part = v[0] * cc[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) part = fmaf(v[j], cc[j], part);
    return part;
}

// Sums R per-lane parts (one per slot) over the L lanes of each row.  The pairs are always
// formed by xor masks L/2, ..., 2, 1 in that order (the tree of a plain butterfly over the row's
// lanes; masks below L never leave the row's group of lanes), but while a lane holds more than
// one slot it hands half of them to its partner at each step ("reduce-scatter"), which needs
// R - 1 + (log2 L - log2 R) shuffles instead of R log2 L.  Each sum is the same IEEE value the
// plain butterfly gives (a + b == b + a exactly), whatever R is.  Afterwards lane l holds the
// total of slot slot_of_lane<R, L>(l) of its row group.
template <int R, int L>
__device__ __forceinline__ float reduce_rows(float (&v)[R], int lane) {
    static_assert(R >= 1 && R <= L && (R & (R - 1)) == 0, "R must be a power of two <= L");
#pragma unroll
    for (int n = R, m = L / 2; n > 1; n >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float give = upper ? v[j] : v[j + n / 2];
            const float keep = upper ? v[j + n / 2] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, give, m);
        }
    }
    float t = v[0];
#pragma unroll
    for (int m = L / (2 * R); m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
    return t;
}

// The slot whose total lane l holds after reduce_rows<R, L>.
template <int R, int L>
__device__ __forceinline__ int slot_of_lane(int lane) {
    int slot = 0;
#pragma unroll
    for (int n = R, m = L / 2; n > 1; n >>= 1, m >>= 1)
        if (lane & m) slot += n / 2;
    return slot;
}

// Lanes that write a readout: one per group of lanes holding the same slot's total.
template <int R, int L>
__device__ __forceinline__ bool writes_row(int lane) {
    return (lane & (L / R - 1)) == 0;
}

// Programmatic dependent launch.  pdl_wait blocks until the grid this one depends on has
// completed and its memory is visible (a no-op when the launch carries no such dependency);
// kernels call it before their first memory access, so a dependent launch never reads or
// writes anything early.  pdl_trigger lets the dependent grid's CTAs start launching.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <bool kIdx64>
__device__ __forceinline__ long long load_slot(const SsuParams &p, long long b) {
    if (kIdx64) return __ldg(static_cast<const long long *>(p.idx) + b * p.idx_s);
    return static_cast<long long>(__ldg(static_cast<const int *>(p.idx) + b * p.idx_s));
}

__device__ __forceinline__ void record_skip(const SsuParams &p, long long b) {
    atomicAdd(&p.err[0], 1u);
    atomicMin(&p.err[1], static_cast<unsigned>(b));
}

}  // namespace
