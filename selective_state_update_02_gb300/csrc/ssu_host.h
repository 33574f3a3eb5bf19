// Host-side pieces shared by the library's translation units: the thread-local error message,
// argument validation and the handle.
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "ssu.h"

namespace ssu_host {

// Records a formatted message for ssu_last_error() and returns `status`.
ssu_status_t fail(ssu_status_t status, const char *fmt, ...);
// Clears the message and returns SSU_OK.
ssu_status_t ok();
bool aligned(const void *ptr, unsigned bytes);
// The full host-side validation of one ssu_update / ssu_update_static call.
ssu_status_t validate_impl(const void *state_pool, const void *idx, const uint16_t *x,
                           const uint16_t *dt, const float *dt_bias, const float *A,
                           const uint16_t *B, const uint16_t *C, const float *D,
                           const uint16_t *out, const ssu_shape_t *shape,
                           const ssu_strides_t *st);

// Rows one warp-wide 16-byte vector instruction covers for this dstate and state type: 1 for
// rows of 512 bytes or more, 2 for 256-byte rows, 4 for 128-byte rows (the kernels' RowGeo).
int rows_per_instruction(int64_t dstate, int32_t state_dtype);
// Whether a kernel instantiation exists for `rows_per_warp` rows per warp: rows_per_instruction
// x {1, 2, 4, 8}, and 16 for an fp32 state of dstate 128.
bool rows_per_warp_ok(int rows_per_warp, int64_t dstate, int32_t state_dtype);

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

}  // namespace ssu_host

struct ssu_handle_s {
    int device = 0;
    int sm_count = 0;
    int smem_optin = 0;       // max dynamic shared memory per CTA (bytes)
    unsigned *err = nullptr;  // device: [0] skipped, [1] smallest skipped request, [2] 0
    bool has_override = false;
    ssu_launch_t override_launch{};
    bool has_copy_override = false;
    ssu_copy_launch_t copy_override{};
    bool pdl = true;  // launch the VEC and multi-token kernels as programmatic dependents
};
