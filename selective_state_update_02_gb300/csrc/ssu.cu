// Mamba2 decode-step selective state update for GB300 (sm_103a): kernels and the C ABI.
//
// The operation and its operands are documented in include/ssu.h (sglang PR #41223,
// Summary and Details / Kernel measurement give the operand set; the arithmetic is the
// standard Mamba2 decode step).  The step is bound by HBM traffic: per (request, head) unit it
// reads and writes a 64 x 128 fp32 state (32 KiB each way) and touches ~2.5 KiB of inputs.
// There is no dense contraction here, so no tensor cores: the design goal is to keep enough
// bytes in flight to saturate HBM3e, with every access a full 16-byte vector per lane.
//
// Work decomposition ("VEC" mode).  A warp owns `RPW` consecutive state rows of one unit;
// lane l owns columns 4l..4l+3 of each row, so each row is one fully coalesced 512-byte
// access per warp and a warp keeps RPW x 512 bytes of loads in flight.  A CTA holds
// `warps_per_cta` such warps over consecutive rows of the same unit.  B[n] and C[n] are read
// straight into registers (each lane needs only its own 4 columns); x[p], dt, dt_bias, A, D
// are warp-uniform broadcast loads.  Each row's readout sum over dstate is the lane's 4-term
// chain followed by a xor-butterfly over the 32 lanes in the fixed mask order 16,8,4,2,1.
// Because that order never depends on RPW or warps_per_cta, every launch shape produces
// bit-identical state and output.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "ssu.h"

namespace {

constexpr int kDstate = 128;  // dstate this build implements: 32 lanes x 4 columns
constexpr int kMaxWarpsPerCta = 16;

// Everything one launch needs, passed by value in the kernel parameter space.
struct SsuParams {
    float *state;
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
    int nheads, headdim, heads_per_group;
    int slabs;         // CTAs per unit
    int rows_per_cta;  // RPW * warps_per_cta
    unsigned *err;     // [0] skipped requests, [1] smallest skipped request index
};

__device__ __forceinline__ float softplus_f32(float z) {
    // log(1 + e^z); above 20 the correction is below fp32 resolution of z.
    return z > 20.0f ? z : log1pf(expf(z));
}

__device__ __forceinline__ float butterfly_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

template <bool kIdx64>
__device__ __forceinline__ long long load_slot(const SsuParams &p, long long b) {
    if (kIdx64) return __ldg(static_cast<const long long *>(p.idx) + b * p.idx_s);
    return static_cast<long long>(__ldg(static_cast<const int *>(p.idx) + b * p.idx_s));
}

template <int RPW, bool kIdx64>
__global__ void __launch_bounds__(32 * kMaxWarpsPerCta)
    ssu_vec_kernel(const __grid_constant__ SsuParams p) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned tile = blockIdx.x;
    const int slab = static_cast<int>(tile % static_cast<unsigned>(p.slabs));
    const unsigned unit = tile / static_cast<unsigned>(p.slabs);
    const int h = static_cast<int>(unit % static_cast<unsigned>(p.nheads));
    const long long b = static_cast<long long>(unit / static_cast<unsigned>(p.nheads));

    const long long s = load_slot<kIdx64>(p, b);
    if (s < 0 || s >= p.pool_size) {
        if (h == 0 && slab == 0 && threadIdx.x == 0) {
            atomicAdd(&p.err[0], 1u);
            atomicMin(&p.err[1], static_cast<unsigned>(b));
        }
        return;
    }

    const int row0 = slab * p.rows_per_cta + warp * RPW;
    float *srow = p.state + s * p.st_pool + h * p.st_head + row0 * p.st_row + lane * 4;

    // Issue every state load of this warp before anything that depends on other loads.
    float4 v[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        if (row0 + r < p.headdim)
            v[r] = __ldcs(reinterpret_cast<const float4 *>(srow + r * p.st_row));
        else
            v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // Per-unit scalars, computed while the state loads are in flight.
    const float z = __bfloat162float(p.dt[b * p.dt_b + h * p.dt_h]) + p.dt_bias[h * p.bias_h];
    const float dtv = softplus_f32(z);
    const float dA = expf(dtv * p.A[h * p.A_h]);
    const float Dh = p.D[h * p.D_h];
    const int g = h / p.heads_per_group;
    const __nv_bfloat16 *Bp = p.B + b * p.B_b + g * p.B_g + lane * 4;
    const __nv_bfloat16 *Cp = p.C + b * p.C_b + g * p.C_g + lane * 4;
    const float b0 = __bfloat162float(Bp[0]), b1 = __bfloat162float(Bp[1]);
    const float b2 = __bfloat162float(Bp[2]), b3 = __bfloat162float(Bp[3]);
    const float c0 = __bfloat162float(Cp[0]), c1 = __bfloat162float(Cp[1]);
    const float c2 = __bfloat162float(Cp[2]), c3 = __bfloat162float(Cp[3]);
    const __nv_bfloat16 *xp = p.x + b * p.x_b + h * p.x_h + row0;

    float mine = 0.f;  // lane r keeps the readout of row row0 + r
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        if (row0 + r < p.headdim) {
            const float xr = __bfloat162float(xp[r]);
            const float k = dtv * xr;
            float4 w = v[r];
            w.x = fmaf(w.x, dA, k * b0);
            w.y = fmaf(w.y, dA, k * b1);
            w.z = fmaf(w.z, dA, k * b2);
            w.w = fmaf(w.w, dA, k * b3);
            __stcs(reinterpret_cast<float4 *>(srow + r * p.st_row), w);
            float part = w.x * c0;
            part = fmaf(w.y, c1, part);
            part = fmaf(w.z, c2, part);
            part = fmaf(w.w, c3, part);
            const float y = fmaf(Dh, xr, butterfly_sum(part));
            if (lane == r) mine = y;
        }
    }
    if (lane < RPW && row0 + lane < p.headdim)
        p.out[b * p.out_b + h * p.out_h + row0 + lane] = __float2bfloat16_rn(mine);
}

template <bool kIdx64>
cudaError_t launch_vec(const SsuParams &p, int rpw, int wpc, unsigned grid, cudaStream_t st) {
    const dim3 block(32 * wpc);
    switch (rpw) {
        case 1: ssu_vec_kernel<1, kIdx64><<<grid, block, 0, st>>>(p); break;
        case 2: ssu_vec_kernel<2, kIdx64><<<grid, block, 0, st>>>(p); break;
        case 4: ssu_vec_kernel<4, kIdx64><<<grid, block, 0, st>>>(p); break;
        case 8: ssu_vec_kernel<8, kIdx64><<<grid, block, 0, st>>>(p); break;
        case 16: ssu_vec_kernel<16, kIdx64><<<grid, block, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Host side: errors, validation, launch-shape table.

thread_local std::string g_last_error;

ssu_status_t fail(ssu_status_t status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

ssu_status_t ok() {
    g_last_error.clear();
    return SSU_OK;
}

bool aligned(const void *ptr, unsigned bytes) {
    return (reinterpret_cast<unsigned long long>(ptr) % bytes) == 0;
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            switched = (err == cudaSuccess);
        }
    }
    ~DeviceGuard() {
        if (switched) cudaSetDevice(prev);
    }
};

ssu_status_t validate_impl(const float *state_pool, const void *idx, const uint16_t *x,
                           const uint16_t *dt, const float *dt_bias, const float *A,
                           const uint16_t *B, const uint16_t *C, const float *D,
                           const uint16_t *out, const ssu_shape_t *shape,
                           const ssu_strides_t *st) {
    if (!shape || !st) return fail(SSU_ERR_INVALID_ARG, "shape and strides must not be NULL");
    const ssu_shape_t &s = *shape;
    if (s.batch < 0) return fail(SSU_ERR_INVALID_ARG, "batch %lld < 0", (long long)s.batch);
    if (s.nheads < 1 || s.headdim < 1 || s.dstate < 1 || s.ngroups < 1)
        return fail(SSU_ERR_INVALID_ARG, "nheads, headdim, dstate and ngroups must be >= 1");
    if (s.pool_size < 0) return fail(SSU_ERR_INVALID_ARG, "pool_size < 0");
    if (s.nheads % s.ngroups != 0)
        return fail(SSU_ERR_INVALID_ARG, "nheads %lld is not a multiple of ngroups %lld",
                    (long long)s.nheads, (long long)s.ngroups);
    if (s.index_dtype != SSU_INDEX_I32 && s.index_dtype != SSU_INDEX_I64)
        return fail(SSU_ERR_INVALID_ARG, "index_dtype %d is neither I32 nor I64", s.index_dtype);
    if (s.dstate != kDstate)
        return fail(SSU_ERR_UNSUPPORTED, "dstate %lld: this build implements dstate 128",
                    (long long)s.dstate);
    if (s.headdim > (1 << 20) || s.nheads > (1 << 20))
        return fail(SSU_ERR_UNSUPPORTED, "headdim and nheads are limited to 2^20");

    const int64_t *all[] = {st->state, st->x, st->out, st->dt, st->B, st->C,
                            st->dt_bias, st->D, st->A};
    const int lens[] = {4, 3, 3, 3, 3, 3, 2, 2, 3};
    for (int i = 0; i < 9; ++i)
        for (int j = 0; j < lens[i]; ++j)
            if (all[i][j] < 0) return fail(SSU_ERR_INVALID_ARG, "negative stride");
    if (st->idx < 0) return fail(SSU_ERR_INVALID_ARG, "negative index stride");
    if (st->state[3] != 1) return fail(SSU_ERR_UNSUPPORTED, "state dstate-stride must be 1");
    if (st->x[2] != 1) return fail(SSU_ERR_UNSUPPORTED, "x headdim-stride must be 1");
    if (st->out[2] != 1) return fail(SSU_ERR_UNSUPPORTED, "out headdim-stride must be 1");
    if (st->B[2] != 1 || st->C[2] != 1)
        return fail(SSU_ERR_UNSUPPORTED, "B and C dstate-stride must be 1");
    if (st->dt[2] != 0) return fail(SSU_ERR_UNSUPPORTED, "dt must be constant over headdim");
    if (st->dt_bias[1] != 0 || st->D[1] != 0)
        return fail(SSU_ERR_UNSUPPORTED, "dt_bias and D must be constant over headdim");
    if (st->A[1] != 0 || st->A[2] != 0)
        return fail(SSU_ERR_UNSUPPORTED, "A must be constant over headdim and dstate");
    for (int j = 0; j < 3; ++j)
        if (st->state[j] % 4 != 0)
            return fail(SSU_ERR_MISALIGNED, "state stride %d (%lld) is not a multiple of 4 floats",
                        j, (long long)st->state[j]);

    if (s.batch == 0) return ok();
    if (!state_pool || !idx || !x || !dt || !dt_bias || !A || !B || !C || !D || !out)
        return fail(SSU_ERR_INVALID_ARG, "a data pointer is NULL");
    if (!aligned(state_pool, 16))
        return fail(SSU_ERR_MISALIGNED, "state_pool is not 16-byte aligned");
    if (!aligned(idx, s.index_dtype == SSU_INDEX_I64 ? 8 : 4))
        return fail(SSU_ERR_MISALIGNED, "state_batch_indices is not aligned to its type");
    if (!aligned(x, 2) || !aligned(dt, 2) || !aligned(B, 2) || !aligned(C, 2) || !aligned(out, 2))
        return fail(SSU_ERR_MISALIGNED, "a bf16 operand is not 2-byte aligned");
    if (!aligned(dt_bias, 4) || !aligned(A, 4) || !aligned(D, 4))
        return fail(SSU_ERR_MISALIGNED, "an fp32 operand is not 4-byte aligned");
    if (s.batch > INT_MAX / s.nheads)
        return fail(SSU_ERR_UNSUPPORTED, "batch * nheads exceeds 2^31");
    return ok();
}

bool launch_shape_ok(const ssu_launch_t &l) {
    if (l.mode != SSU_MODE_VEC) return false;
    const int r = l.rows_per_warp;
    if (r != 1 && r != 2 && r != 4 && r != 8 && r != 16) return false;
    return l.warps_per_cta >= 1 && l.warps_per_cta <= kMaxWarpsPerCta;
}

// Built-in launch-shape table.  8 rows per warp (32 floats, 128 bytes of loads in flight
// per thread) with few warps per CTA; the CTA count then spreads small batches over all SMs.
ssu_launch_t table_launch(const ssu_shape_t &s, int sm_count) {
    ssu_launch_t l{SSU_MODE_VEC, 8, 1, 0};
    const long long rows = s.batch * s.nheads * s.headdim;
    const long long warps_needed = (rows + 7) / 8;
    // Batches large enough to give every SM many warps use 2-warp CTAs.
    if (warps_needed >= 16LL * sm_count) l.warps_per_cta = 2;
    return l;
}

}  // namespace

struct ssu_handle_s {
    int device = 0;
    int sm_count = 0;
    unsigned *err = nullptr;  // device: [0] skipped count, [1] smallest skipped request
    bool has_override = false;
    ssu_launch_t override_launch{};
};

extern "C" {

int32_t ssu_abi_version(void) { return SSU_ABI_VERSION; }

const char *ssu_status_string(ssu_status_t status) {
    switch (status) {
        case SSU_OK: return "SSU_OK";
        case SSU_ERR_INVALID_ARG: return "SSU_ERR_INVALID_ARG";
        case SSU_ERR_UNSUPPORTED: return "SSU_ERR_UNSUPPORTED";
        case SSU_ERR_MISALIGNED: return "SSU_ERR_MISALIGNED";
        case SSU_ERR_CUDA: return "SSU_ERR_CUDA";
        case SSU_ERR_INDEX_OOB: return "SSU_ERR_INDEX_OOB";
    }
    return "SSU_ERR_UNKNOWN";
}

const char *ssu_last_error(void) { return g_last_error.c_str(); }

ssu_status_t ssu_create(ssu_handle_t *out, int32_t device) {
    if (!out) return fail(SSU_ERR_INVALID_ARG, "out must not be NULL");
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess || device < 0 || device >= count)
        return fail(SSU_ERR_CUDA, "no CUDA device %d (%s)", device,
                    e == cudaSuccess ? "out of range" : cudaGetErrorString(e));
    DeviceGuard guard(device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    ssu_handle_s *h = new ssu_handle_s();
    h->device = device;
    e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaMalloc(&h->err, 4 * sizeof(unsigned));
    const unsigned init[4] = {0u, 0xffffffffu, 0u, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(h->err, init, sizeof(init), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (h->err) cudaFree(h->err);
        delete h;
        return fail(SSU_ERR_CUDA, "ssu_create: %s", cudaGetErrorString(e));
    }
    *out = h;
    return ok();
}

ssu_status_t ssu_destroy(ssu_handle_t handle) {
    if (!handle) return ok();
    ssu_status_t st = SSU_OK;
    {
        DeviceGuard guard(handle->device);
        if (handle->err && cudaFree(handle->err) != cudaSuccess) st = SSU_ERR_CUDA;
    }
    delete handle;
    return st == SSU_OK ? ok() : fail(st, "cudaFree failed in ssu_destroy");
}

ssu_status_t ssu_validate(const float *state_pool, const void *state_batch_indices,
                          const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                          const float *A, const uint16_t *B, const uint16_t *C, const float *D,
                          const uint16_t *out, const ssu_shape_t *shape,
                          const ssu_strides_t *strides) {
    return validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D, out, shape,
                         strides);
}

ssu_status_t ssu_get_launch(ssu_handle_t handle, const ssu_shape_t *shape,
                            ssu_launch_t *launch) {
    if (!handle || !shape || !launch) return fail(SSU_ERR_INVALID_ARG, "NULL argument");
    *launch = handle->has_override ? handle->override_launch
                                   : table_launch(*shape, handle->sm_count);
    return ok();
}

ssu_status_t ssu_set_launch(ssu_handle_t handle, const ssu_launch_t *launch) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    if (!launch || launch->mode == SSU_MODE_AUTO) {
        handle->has_override = false;
        return ok();
    }
    if (!launch_shape_ok(*launch))
        return fail(SSU_ERR_UNSUPPORTED, "launch shape mode=%d rows_per_warp=%d warps=%d",
                    launch->mode, launch->rows_per_warp, launch->warps_per_cta);
    handle->override_launch = *launch;
    handle->has_override = true;
    return ok();
}

ssu_status_t ssu_update(ssu_handle_t handle, float *state_pool, const void *state_batch_indices,
                        const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                        const float *A, const uint16_t *B, const uint16_t *C, const float *D,
                        uint16_t *out, const ssu_shape_t *shape, const ssu_strides_t *strides,
                        ssu_stream_t stream) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    ssu_status_t st = validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                                    D, out, shape, strides);
    if (st != SSU_OK || shape->batch == 0) return st;
    const ssu_shape_t &s = *shape;
    const ssu_launch_t l = handle->has_override ? handle->override_launch
                                                : table_launch(s, handle->sm_count);
    const int rows_per_cta = l.rows_per_warp * l.warps_per_cta;
    const long long slabs = (s.headdim + rows_per_cta - 1) / rows_per_cta;
    const long long grid = s.batch * s.nheads * slabs;
    if (grid > INT_MAX) return fail(SSU_ERR_UNSUPPORTED, "grid of %lld CTAs exceeds 2^31", grid);

    SsuParams p;
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
    p.nheads = static_cast<int>(s.nheads);
    p.headdim = static_cast<int>(s.headdim);
    p.heads_per_group = static_cast<int>(s.nheads / s.ngroups);
    p.slabs = static_cast<int>(slabs);
    p.rows_per_cta = rows_per_cta;
    p.err = handle->err;

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        s.index_dtype == SSU_INDEX_I64
            ? launch_vec<true>(p, l.rows_per_warp, l.warps_per_cta, (unsigned)grid, cs)
            : launch_vec<false>(p, l.rows_per_warp, l.warps_per_cta, (unsigned)grid, cs);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ok();
}

ssu_status_t ssu_get_error(ssu_handle_t handle, ssu_stream_t stream, uint32_t *skipped,
                           int64_t *first_bad) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    unsigned host[2] = {0u, 0xffffffffu};
    if (e == cudaSuccess) e = cudaMemcpy(host, handle->err, sizeof(host), cudaMemcpyDeviceToHost);
    const unsigned init[2] = {0u, 0xffffffffu};
    if (e == cudaSuccess) e = cudaMemcpy(handle->err, init, sizeof(init), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "ssu_get_error: %s", cudaGetErrorString(e));
    if (skipped) *skipped = host[0];
    if (first_bad) *first_bad = host[0] ? static_cast<int64_t>(host[1]) : -1;
    if (host[0]) return fail(SSU_ERR_INDEX_OOB, "%u request(s) named a slot outside the pool",
                             host[0]);
    return ok();
}

}  // extern "C"
