// Device-side pieces shared by the decode-step kernels: launch constants, the parameter block,
// the per-element arithmetic, the readout reduction, slot lookup, and the mbarrier / bulk-copy
// PTX wrappers.  Included by each kernel translation unit (internal linkage per unit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kDstate = 128;             // dstate of the BULK kernel: 32 lanes x 4 columns
constexpr int kRowBytes = kDstate * 4;   // one fp32 state row of the BULK kernel
constexpr int kMaxWarpsPerCta = 16;      // VEC
constexpr int kMaxBulkWarps = 8;         // BULK compute warps (plus one producer warp)
constexpr int kMaxStages = 8;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per mbarrier wait

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
    unsigned *err;     // [0] skipped requests, [1] smallest skipped request, [2] timeouts
};

// BULK launch geometry.
struct BulkShape {
    long long tiles;  // batch * nheads * slabs
    int stages;
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

// The update of one lane's 4 columns of one row; returns the lane's part of the readout.
__device__ __forceinline__ float update_cols(float4 &w, float dA, float k, const float (&bb)[4],
                                             const float (&cc)[4]) {
    w.x = fmaf(w.x, dA, k * bb[0]);
    w.y = fmaf(w.y, dA, k * bb[1]);
    w.z = fmaf(w.z, dA, k * bb[2]);
    w.w = fmaf(w.w, dA, k * bb[3]);
    float part = w.x * cc[0];
    part = fmaf(w.y, cc[1], part);
    part = fmaf(w.z, cc[2], part);
    part = fmaf(w.w, cc[3], part);
    return part;
}

// ---------------------------------------------------------------------------------------
// Columns of a row owned by one lane, for dstate N = 32 * NC (NC = 2, 4 or 8).  With NC = 2
// lane l owns columns 2l, 2l+1; with NC = 4 columns 4l..4l+3; with NC = 8 the two groups
// 4l..4l+3 and 128+4l..128+4l+3, so every vector instruction of a warp covers one contiguous
// span of the row.  The lane's j-th value is column lane_offset<NC>(lane) + (j / 4) * 128 +
// j % 4.

// Offset of a lane's first column in a row (its columns then sit at +0..3 and, for NC = 8,
// +128..131; for NC = 2 at +0..1).  Kernels add it to the row pointer once.
template <int NC>
__device__ __forceinline__ int lane_offset(int lane) {
    return NC == 2 ? 2 * lane : 4 * lane;
}

__device__ __forceinline__ float2 bf2_to_f2(unsigned bits) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bits));
}

__device__ __forceinline__ unsigned f2_to_bf2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // round to nearest even
    return *reinterpret_cast<const unsigned *>(&h);
}

// Streaming (evict-first) load of one lane's NC columns of a row, widened to fp32.  `p` points
// at the lane's first column (row + lane_offset<NC>(lane)).
template <int NC, typename ST>
__device__ __forceinline__ void load_cols(const ST *p, float (&v)[NC]) {
    if constexpr (sizeof(ST) == 4) {
        if constexpr (NC == 2) {
            const float2 a = __ldcs(reinterpret_cast<const float2 *>(p));
            v[0] = a.x, v[1] = a.y;
        } else {
#pragma unroll
            for (int g = 0; g < NC / 4; ++g) {
                const float4 a = __ldcs(reinterpret_cast<const float4 *>(p + g * 128));
                v[4 * g] = a.x, v[4 * g + 1] = a.y, v[4 * g + 2] = a.z, v[4 * g + 3] = a.w;
            }
        }
    } else {
        if constexpr (NC == 2) {
            const float2 a = bf2_to_f2(__ldcs(reinterpret_cast<const unsigned *>(p)));
            v[0] = a.x, v[1] = a.y;
        } else {
#pragma unroll
            for (int g = 0; g < NC / 4; ++g) {
                const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p + g * 128));
                const float2 a = bf2_to_f2(u.x), b = bf2_to_f2(u.y);
                v[4 * g] = a.x, v[4 * g + 1] = a.y, v[4 * g + 2] = b.x, v[4 * g + 3] = b.y;
            }
        }
    }
}

// Streaming store of one lane's NC columns (rounded to bf16, nearest even, for a bf16 state);
// `p` points at the lane's first column.
template <int NC, typename ST>
__device__ __forceinline__ void store_cols(ST *p, const float (&v)[NC]) {
    if constexpr (sizeof(ST) == 4) {
        if constexpr (NC == 2) {
            __stcs(reinterpret_cast<float2 *>(p), make_float2(v[0], v[1]));
        } else {
#pragma unroll
            for (int g = 0; g < NC / 4; ++g)
                __stcs(reinterpret_cast<float4 *>(p + g * 128),
                       make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
        }
    } else {
        if constexpr (NC == 2) {
            __stcs(reinterpret_cast<unsigned *>(p), f2_to_bf2(v[0], v[1]));
        } else {
#pragma unroll
            for (int g = 0; g < NC / 4; ++g)
                __stcs(reinterpret_cast<uint2 *>(p + g * 128),
                       make_uint2(f2_to_bf2(v[4 * g], v[4 * g + 1]),
                                  f2_to_bf2(v[4 * g + 2], v[4 * g + 3])));
        }
    }
}

// The lane's NC columns of B (or C), widened to fp32; `p` points at the lane's first column.
template <int NC>
__device__ __forceinline__ void load_bc(const __nv_bfloat16 *p, float (&o)[NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) o[j] = __bfloat162float(p[(j / 4) * 128 + (j % 4)]);
}

// The update of one lane's NC columns of one row; returns the lane's part of the readout
// (its columns summed in order j = 0, 1, ...); for NC = 4 the same operations as update_cols.
template <int NC>
__device__ __forceinline__ float update_lane(float (&v)[NC], float dA, float k,
                                             const float (&bb)[NC], const float (&cc)[NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) v[j] = fmaf(v[j], dA, k * bb[j]);
    float part = v[0] * cc[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) part = fmaf(v[j], cc[j], part);
    return part;
}

// Sums R per-lane parts (one per row) over the 32 lanes.  The pairs are always formed by xor
// masks 16, 8, 4, 2, 1 in that order (the tree of a plain butterfly), but while a lane holds
// more than one row it hands half of its rows to its partner at each step ("reduce-scatter"),
// which needs R - 1 + (5 - log2 R) shuffles instead of 5 R.  Each sum is the same IEEE value the
// plain butterfly gives (a + b == b + a exactly), whatever R is.  Afterwards lane l holds the
// total of row row_of_lane<R>(l).
template <int R>
__device__ __forceinline__ float reduce_rows(float (&v)[R], int lane) {
    static_assert(R >= 1 && R <= 32 && (R & (R - 1)) == 0, "R must be a power of two <= 32");
#pragma unroll
    for (int n = R, m = 16; n > 1; n >>= 1, m >>= 1) {
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
    for (int m = 16 / R; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
    return t;
}

// The row whose total lane l holds after reduce_rows<R>.
template <int R>
__device__ __forceinline__ int row_of_lane(int lane) {
    int row = 0;
#pragma unroll
    for (int n = R, m = 16; n > 1; n >>= 1, m >>= 1)
        if (lane & m) row += n / 2;
    return row;
}

// Lanes that write a readout: one per group of lanes holding the same row.
template <int R>
__device__ __forceinline__ bool writes_row(int lane) {
    return (lane & (32 / R - 1)) == 0;
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

// ---------------------------------------------------------------------------------------
// BULK kernel: PTX helpers (mbarrier, bulk asynchronous copies, proxy fence)

__device__ __forceinline__ unsigned smem_u32(const void *ptr) {
    return static_cast<unsigned>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete; false after kWaitLimitNs without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 32; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, unsigned bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

}  // namespace
