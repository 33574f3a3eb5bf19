// Mamba2 decode-step selective state update for GB300 (sm_103a): the single-step C ABI
// (handles, validation, launch table, ssu_update, error counters, the allocation-free entry).
//
// The operation and its operands are documented in include/ssu.h (sglang PR #41223,
// Summary and Details / Kernel measurement give the operand set; the arithmetic is the
// standard Mamba2 decode step).  The step is bound by HBM traffic: per (request, head) unit it
// reads and writes a 64 x 128 fp32 state (32 KiB each way) and touches ~2.5 KiB of inputs.
// There is no dense contraction here, so no tensor cores.
//
// One kernel computes it (ssu_vec.cuh): one CTA per (slab of rows, head, request); each warp
// holds its rows in registers, 16-byte vector loads all issued before any use.  Every launch
// shape gives bit-identical state and output (one fixed summation order per row).
// The multi-token step and the state-block copy live in ssu_tokens.cu and ssu_copy.cu.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cctype>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "ssu.h"
#include "ssu_device.cuh"
#include "ssu_stage.cuh"
#include "ssu_vec.cuh"
#include "ssu_host.h"

using ssu_host::aligned;
using ssu_host::DeviceGuard;
using ssu_host::fail;
using ssu_host::ok;
using ssu_host::validate_impl;

namespace {


// Checks a launch shape by itself (sizes some bucket accepts); rows_per_warp_ok checks it
// against the call's dstate and state type.
bool launch_shape_ok(const ssu_launch_t &l) {
    const int r = l.rows_per_warp;
    return l.mode == SSU_MODE_VEC && r >= 1 && r <= 32 && (r & (r - 1)) == 0 &&
           l.warps_per_cta >= 1 && l.warps_per_cta <= kMaxWarpsPerCta;
}

// Parses a launch spec: NULL, "", "auto" (the table), or "[vec,]rows_per_warp,warps_per_cta"
// with optional spaces.  Only the syntax is checked here; ssu_set_launch checks the shape.
ssu_status_t parse_launch_spec(const char *spec, ssu_launch_t *out) {
    *out = ssu_launch_t{SSU_MODE_AUTO, 0, 0, 0};
    if (!spec) return ok();
    char buf[64];
    size_t n = 0;
    for (const char *c = spec; *c; ++c) {
        if (*c == ' ' || *c == '\t') continue;
        if (n + 1 >= sizeof(buf)) return fail(SSU_ERR_INVALID_ARG, "launch spec too long");
        buf[n++] = static_cast<char>(tolower(static_cast<unsigned char>(*c)));
    }
    buf[n] = 0;
    if (n == 0 || strcmp(buf, "auto") == 0) return ok();
    const char *q = buf;
    if (strncmp(q, "vec,", 4) == 0) q += 4;
    int vals[2];
    for (int i = 0; i < 2; ++i) {
        if (*q < '0' || *q > '9')
            return fail(SSU_ERR_INVALID_ARG, "launch spec '%s': expected [vec,]rows,warps", spec);
        long v = 0;
        while (*q >= '0' && *q <= '9') {
            v = v * 10 + (*q++ - '0');
            if (v > 1024)
                return fail(SSU_ERR_INVALID_ARG, "launch spec '%s': value too large", spec);
        }
        vals[i] = static_cast<int>(v);
        if (i == 0 && *q++ != ',')
            return fail(SSU_ERR_INVALID_ARG, "launch spec '%s': expected [vec,]rows,warps", spec);
    }
    if (*q)
        return fail(SSU_ERR_INVALID_ARG, "launch spec '%s': trailing characters", spec);
    *out = ssu_launch_t{SSU_MODE_VEC, vals[0], vals[1], 0};
    return ok();
}

}  // namespace

namespace {

// Built-in launch-shape table, from the cold-L2 sweeps on GB300 (bench.py --sweep with and
// without --dstate / --state-dtype, batch 8, 128 and 512 at 16 heads, headdim 64), keyed by
// the bytes of one state row.  A warp's unit of work is a vector row ("slot"): the rows one
// 16-byte-per-lane instruction covers (1 row of 512 B, 2 of 256 B, 4 of 128 B; a 1 KiB row
// takes two vectors per lane).  Call sizes are state bytes per call, scaled to 152 SMs.
//   1 KiB rows:  4 slots x 2 warps from 16 MiB, else 2 x 4.
//   512 B rows:  8 slots x 4 warps (x 2 for bf16) from 8 MiB (batch 16 at 16 heads of 64 rows),
//                else 2 x 4.  16 rows per warp is slower in every bucket.
//   256 B rows:  8 slots x 4 warps from 8 MiB, else 4 x 4 (fp32 dstate 64, batch 8: 3.14 us at
//                2 slots, 2.62 at 4).
//   128 B rows:  8 slots x 2 warps from 32 MiB, 4 x 4 from 8 MiB (batch 128: 8.19 us at 8 x 2,
//                7.84 at 4 x 4), else 2 x 8.
// The tile never exceeds the headdim.
ssu_launch_t table_launch(const ssu_handle_s &hd, const ssu_shape_t &s, const ssu_strides_t *st) {
    (void)st;
    const bool bf16 = s.state_dtype == SSU_STATE_BF16;
    const long long row_bytes = s.dstate * (bf16 ? 2 : 4);
    const int rpi = ssu_host::rows_per_instruction(s.dstate, s.state_dtype);
    const long long bytes = s.batch * s.nheads * s.headdim * row_bytes;
    auto at_least = [&](long long mib) { return bytes * 152 >= (mib << 20) * hd.sm_count; };
    int slots, wpc;
    if (row_bytes >= 1024) {
        slots = at_least(16) ? 4 : 2;
        wpc = at_least(16) ? 2 : 4;
    } else if (row_bytes == 512) {
        slots = at_least(8) ? 8 : 2;
        wpc = at_least(8) && bf16 ? 2 : 4;
    } else if (row_bytes == 256) {
        slots = at_least(8) ? 8 : 4;
        wpc = 4;
    } else {
        slots = at_least(32) ? 8 : at_least(8) ? 4 : 2;
        wpc = at_least(32) ? 2 : at_least(8) ? 4 : 8;
    }
    int rpw = slots * rpi;
    while (slots > 1 && rpw > s.headdim) {
        slots >>= 1;
        rpw = slots * rpi;
    }
    while (wpc > 1 && rpw * wpc > s.headdim) wpc >>= 1;
    return ssu_launch_t{SSU_MODE_VEC, rpw, wpc, 0};
}

// The kernels' parameter block for one call (validated arguments, element strides).
SsuParams make_params(void *state_pool, const void *idx, const uint16_t *x, const uint16_t *dt,
                      const float *dt_bias, const float *A, const uint16_t *B, const uint16_t *C,
                      const float *D, uint16_t *out, const ssu_shape_t &s,
                      const ssu_strides_t *strides, long long slabs, int rows_per_tile,
                      unsigned *err) {
    SsuParams p;
    p.state = state_pool;
    p.idx = idx;
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
    p.err = err;
    return p;
}

}  // namespace

extern "C" {

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
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   device);
    if (e == cudaSuccess) e = cudaMalloc(&h->err, 4 * sizeof(unsigned));
    const unsigned init[4] = {0u, 0xffffffffu, 0u, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(h->err, init, sizeof(init), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (h->err) cudaFree(h->err);
        delete h;
        return fail(SSU_ERR_CUDA, "ssu_create: %s", cudaGetErrorString(e));
    }
    // SSU_LAUNCH in the environment: the handle's initial launch override.
    if (const char *env = getenv("SSU_LAUNCH")) {
        const ssu_status_t st = ssu_set_launch_override(h, env);
        if (st != SSU_OK) {
            cudaFree(h->err);
            delete h;
            return st;
        }
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

ssu_status_t ssu_validate(const void *state_pool, const void *state_batch_indices,
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
                                   : table_launch(*handle, *shape, nullptr);
    return ok();
}

ssu_status_t ssu_set_launch(ssu_handle_t handle, const ssu_launch_t *launch) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    if (!launch || launch->mode == SSU_MODE_AUTO) {
        handle->has_override = false;
        return ok();
    }
    if (!launch_shape_ok(*launch))
        return fail(SSU_ERR_UNSUPPORTED,
                    "launch shape mode=%d rows_per_warp=%d warps=%d stages=%d", launch->mode,
                    launch->rows_per_warp, launch->warps_per_cta, launch->stages);
    handle->override_launch = *launch;
    handle->has_override = true;
    return ok();
}

ssu_status_t ssu_set_launch_override(ssu_handle_t handle, const char *spec) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    ssu_launch_t l{};
    const ssu_status_t st = parse_launch_spec(spec, &l);
    if (st != SSU_OK) return st;
    return ssu_set_launch(handle, l.mode == SSU_MODE_AUTO ? nullptr : &l);
}

ssu_status_t ssu_set_pdl(ssu_handle_t handle, int32_t enable) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    handle->pdl = enable != 0;
    return ok();
}

ssu_status_t ssu_update(ssu_handle_t handle, void *state_pool, const void *state_batch_indices,
                        const uint16_t *x, const uint16_t *dt, const float *dt_bias,
                        const float *A, const uint16_t *B, const uint16_t *C, const float *D,
                        uint16_t *out, const ssu_shape_t *shape, const ssu_strides_t *strides,
                        ssu_stream_t stream) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    ssu_status_t st = validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                                    D, out, shape, strides);
    if (st != SSU_OK || shape->batch == 0) return st;
    const ssu_shape_t &s = *shape;
    ssu_launch_t l = handle->has_override ? handle->override_launch
                                          : table_launch(*handle, s, strides);
    if (!ssu_host::rows_per_warp_ok(l.rows_per_warp, s.dstate, s.state_dtype))
        return fail(SSU_ERR_UNSUPPORTED,
                    "%d rows per warp: dstate %lld with a %s state takes %d x {1, 2, 4, 8}%s",
                    l.rows_per_warp, (long long)s.dstate,
                    s.state_dtype == SSU_STATE_BF16 ? "bf16" : "fp32",
                    ssu_host::rows_per_instruction(s.dstate, s.state_dtype),
                    s.dstate == 128 && s.state_dtype == SSU_STATE_F32 ? " or 16" : "");
    const int rows_per_tile = l.rows_per_warp * l.warps_per_cta;
    const long long slabs = (s.headdim + rows_per_tile - 1) / rows_per_tile;
    const long long tiles = s.batch * s.nheads * slabs;
    if (tiles > INT_MAX)
        return fail(SSU_ERR_UNSUPPORTED, "%lld tiles exceed 2^31", tiles);

    const SsuParams p = make_params(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                                    out, s, strides, slabs, rows_per_tile, handle->err);

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool i64 = s.index_dtype == SSU_INDEX_I64;
    const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                    static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535));
    const cudaError_t e =
        launch_vec(p, static_cast<int>(s.dstate), s.state_dtype == SSU_STATE_BF16, i64,
                   l.rows_per_warp, l.warps_per_cta, grid, handle->pdl, cs);
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
    unsigned host[3] = {0u, 0xffffffffu, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(host, handle->err, sizeof(host), cudaMemcpyDeviceToHost);
    const unsigned init[3] = {0u, 0xffffffffu, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(handle->err, init, sizeof(init), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "ssu_get_error: %s", cudaGetErrorString(e));
    if (skipped) *skipped = host[0];
    if (first_bad) *first_bad = host[0] ? static_cast<int64_t>(host[1]) : -1;
    if (host[0]) return fail(SSU_ERR_INDEX_OOB, "%u request(s) named a slot outside the pool",
                             host[0]);
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Per-step operands in host memory: a staging kernel, then the decode-step kernel.

namespace {

long long round256(long long v) { return (v + 255) & ~255LL; }

// Byte offsets of the dense staged operands in the workspace.
struct HostLayout {
    long long idx, x, dt, B, C, total;
};

HostLayout host_layout(const ssu_shape_t &s) {
    const long long esz = s.index_dtype == SSU_INDEX_I64 ? 8 : 4;
    const long long bc = round256(s.batch * s.ngroups * s.dstate * 2);
    HostLayout L;
    L.idx = 0;
    L.x = round256(s.batch * esz);
    L.dt = L.x + round256(s.batch * s.nheads * s.headdim * 2);
    L.B = L.dt + round256(s.batch * s.nheads * 2);
    L.C = L.B + bc;
    L.total = L.C + bc;
    return L;
}

// The address through which kernels on the current device reach operand `p`: the device
// mapping of page-locked host memory, or the pointer itself for device memory of this device
// and for managed memory.
ssu_status_t device_view(const void *p, const char *name, int dev, const void **view) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SSU_ERR_CUDA, "cudaPointerGetAttributes(%s): %s", name,
                    cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeHost) {
        if (!a.devicePointer)
            return fail(SSU_ERR_INVALID_ARG, "%s: page-locked memory not mapped on device %d",
                        name, dev);
        *view = a.devicePointer;
        return SSU_OK;
    }
    if (a.type == cudaMemoryTypeManaged || (a.type == cudaMemoryTypeDevice && a.device == dev)) {
        *view = p;
        return SSU_OK;
    }
    if (a.type == cudaMemoryTypeDevice)
        return fail(SSU_ERR_INVALID_ARG, "%s is memory of device %d, not %d", name, a.device,
                    dev);
    return fail(SSU_ERR_INVALID_ARG,
                "%s is pageable host memory: allocate it with cudaHostAlloc or register it "
                "with cudaHostRegister",
                name);
}

}  // namespace

extern "C" {

ssu_status_t ssu_host_workspace_bytes(const ssu_shape_t *shape, int64_t *bytes) {
    if (!shape || !bytes) return fail(SSU_ERR_INVALID_ARG, "NULL argument");
    const ssu_shape_t &s = *shape;
    if (s.batch < 0 || s.nheads < 1 || s.headdim < 1 || s.dstate < 1 || s.ngroups < 1)
        return fail(SSU_ERR_INVALID_ARG, "batch must be >= 0 and every dimension >= 1");
    *bytes = host_layout(s).total;
    return ok();
}

ssu_status_t ssu_update_from_host(ssu_handle_t handle, void *state_pool,
                                  const void *state_batch_indices, const uint16_t *x,
                                  const uint16_t *dt, const float *dt_bias, const float *A,
                                  const uint16_t *B, const uint16_t *C, const float *D,
                                  uint16_t *out, const ssu_shape_t *shape,
                                  const ssu_strides_t *strides, void *workspace,
                                  int64_t workspace_bytes, ssu_stream_t stream) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    ssu_status_t st = validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                                    D, out, shape, strides);
    if (st != SSU_OK || shape->batch == 0) return st;
    const ssu_shape_t &s = *shape;
    const HostLayout L = host_layout(s);
    if (!workspace) return fail(SSU_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(workspace, 256))
        return fail(SSU_ERR_MISALIGNED, "workspace is not 256-byte aligned");
    if (workspace_bytes < L.total)
        return fail(SSU_ERR_INVALID_ARG, "workspace holds %lld bytes; this shape needs %lld",
                    (long long)workspace_bytes, L.total);
    ssu_launch_t l = handle->has_override && handle->override_launch.mode == SSU_MODE_VEC
                         ? handle->override_launch
                         : table_launch(*handle, s, strides);
    if (!ssu_host::rows_per_warp_ok(l.rows_per_warp, s.dstate, s.state_dtype))
        return fail(SSU_ERR_UNSUPPORTED, "%d rows per warp do not fit dstate %lld",
                    l.rows_per_warp, (long long)s.dstate);
    const int rows_per_tile = l.rows_per_warp * l.warps_per_cta;
    const long long slabs = (s.headdim + rows_per_tile - 1) / rows_per_tile;
    const long long tiles = s.batch * s.nheads * slabs;
    if (tiles > INT_MAX) return fail(SSU_ERR_UNSUPPORTED, "%lld tiles exceed 2^31", tiles);

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    const void *v_idx, *v_x, *v_dt, *v_B, *v_C, *v_out;
    if ((st = device_view(state_batch_indices, "state_batch_indices", handle->device, &v_idx)) ||
        (st = device_view(x, "x", handle->device, &v_x)) ||
        (st = device_view(dt, "dt", handle->device, &v_dt)) ||
        (st = device_view(B, "B", handle->device, &v_B)) ||
        (st = device_view(C, "C", handle->device, &v_C)) ||
        (st = device_view(out, "out", handle->device, &v_out)))
        return st;

    // Dense staged copies: idx [bs], x [bs,H,P], dt [bs,H], B and C [bs,G,N].
    char *ws = static_cast<char *>(workspace);
    const long long esz = s.index_dtype == SSU_INDEX_I64 ? 8 : 4;
    const ssu_strides_t &u = *strides;
    StageParams q;
    long long chunk0 = 0;
    q.job[0] = stage_job(v_idx, ws + L.idx, s.batch, 1, u.idx * esz, 0, esz, chunk0);
    q.job[1] = stage_job(v_x, ws + L.x, s.batch, s.nheads, u.x[0] * 2, u.x[1] * 2,
                         s.headdim * 2, chunk0);
    q.job[2] = stage_job(v_dt, ws + L.dt, s.batch, s.nheads, u.dt[0] * 2, u.dt[1] * 2, 2, chunk0);
    q.job[3] = stage_job(v_B, ws + L.B, s.batch, s.ngroups, u.B[0] * 2, u.B[1] * 2,
                         s.dstate * 2, chunk0);
    q.job[4] = stage_job(v_C, ws + L.C, s.batch, s.ngroups, u.C[0] * 2, u.C[1] * 2,
                         s.dstate * 2, chunk0);
    q.njobs = kStageJobs;
    q.total = chunk0;

    ssu_strides_t dense = u;
    dense.idx = 1;
    const int64_t x_dense[3] = {s.nheads * s.headdim, s.headdim, 1};
    const int64_t dt_dense[3] = {s.nheads, 1, 0};
    const int64_t bc_dense[3] = {s.ngroups * s.dstate, s.dstate, 1};
    for (int i = 0; i < 3; ++i) {
        dense.x[i] = x_dense[i];
        dense.dt[i] = dt_dense[i];
        dense.B[i] = bc_dense[i];
        dense.C[i] = bc_dense[i];
    }
    auto bf = [](const char *ptr) { return reinterpret_cast<const uint16_t *>(ptr); };
    const SsuParams p =
        make_params(state_pool, ws + L.idx, bf(ws + L.x), bf(ws + L.dt), dt_bias, A,
                    bf(ws + L.B), bf(ws + L.C), D,
                    const_cast<uint16_t *>(static_cast<const uint16_t *>(v_out)), s, &dense,
                    slabs, rows_per_tile, handle->err);

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_stage(q, handle->sm_count, handle->pdl, cs);
    if (e == cudaSuccess)
        e = launch_vec(p, static_cast<int>(s.dstate), s.state_dtype == SSU_STATE_BF16,
                       s.index_dtype == SSU_INDEX_I64, l.rows_per_warp, l.warps_per_cta,
                       dim3(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                            static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535)),
                       true, cs);
    if (e != cudaSuccess)
        return fail(SSU_ERR_CUDA, "ssu_update_from_host: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free entry point: the kernel's counters live in a fixed device array.

static __device__ __align__(256) unsigned ssu_static_scratch[SSU_STATIC_SCRATCH_BYTES / 4];

namespace {

// Device address of the array and the SM count of the current device `dev`.  Looked up on
// every call rather than cached: the address belongs to the device's current context, which
// a device reset replaces (the lookup is a host-side table read once the library's module is
// loaded on the device; the first call on a device loads it).
ssu_status_t static_scratch_on(int dev, unsigned **addr, int *sms) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, ssu_static_scratch);
    if (e != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    *addr = static_cast<unsigned *>(ptr);
    *sms = n;
    return SSU_OK;
}

}  // namespace

extern "C" ssu_status_t ssu_update_static(void *state_pool, const void *state_batch_indices,
                                          const uint16_t *x, const uint16_t *dt,
                                          const float *dt_bias, const float *A,
                                          const uint16_t *B, const uint16_t *C, const float *D,
                                          uint16_t *out, const ssu_shape_t *shape,
                                          const ssu_strides_t *strides, uint32_t *counters_out,
                                          ssu_stream_t stream) {
    if (shape && shape->batch > SSU_STATIC_MAX_BATCH)
        return fail(SSU_ERR_UNSUPPORTED,
                    "batch %lld exceeds SSU_STATIC_MAX_BATCH (%lld): the static counters keep "
                    "the smallest skipped request in 32 bits",
                    (long long)shape->batch, (long long)SSU_STATIC_MAX_BATCH);
    ssu_status_t st = validate_impl(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C,
                                    D, out, shape, strides);
    if (st != SSU_OK || shape->batch == 0) return st;
    if (counters_out && !aligned(counters_out, 4))
        return fail(SSU_ERR_MISALIGNED, "counters_out is not 4-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    unsigned *scratch = nullptr;
    int sms = 0;
    st = static_scratch_on(dev, &scratch, &sms);
    if (st != SSU_OK) return st;

    const ssu_shape_t &s = *shape;
    ssu_handle_s table_only;
    table_only.sm_count = sms;
    ssu_launch_t l = table_launch(table_only, s, strides);
    const int rows_per_tile = l.rows_per_warp * l.warps_per_cta;
    const long long slabs = (s.headdim + rows_per_tile - 1) / rows_per_tile;
    const long long tiles = s.batch * s.nheads * slabs;
    if (tiles > INT_MAX) return fail(SSU_ERR_UNSUPPORTED, "%lld tiles exceed 2^31", tiles);

    const SsuParams p = make_params(state_pool, state_batch_indices, x, dt, dt_bias, A, B, C, D,
                                    out, s, strides, slabs, rows_per_tile, scratch);

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // The counters start every call at {0 skipped, no smallest index (all ones), 0 (reserved)}.
    e = cudaMemsetAsync(scratch, 0, 3 * sizeof(unsigned), cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch + 1, 0xff, sizeof(unsigned), cs);
    if (e == cudaSuccess)
        e = launch_vec(p, static_cast<int>(s.dstate), s.state_dtype == SSU_STATE_BF16,
                       s.index_dtype == SSU_INDEX_I64, l.rows_per_warp, l.warps_per_cta,
                       dim3(static_cast<unsigned>(slabs), static_cast<unsigned>(s.nheads),
                            static_cast<unsigned>(s.batch < 65535 ? s.batch : 65535)),
                       false, cs);
    if (e == cudaSuccess && counters_out)
        e = cudaMemcpyAsync(counters_out, scratch, 3 * sizeof(unsigned),
                            cudaMemcpyDeviceToDevice, cs);
    if (e != cudaSuccess)
        return fail(SSU_ERR_CUDA, "ssu_update_static: %s", cudaGetErrorString(e));
    return ok();
}
