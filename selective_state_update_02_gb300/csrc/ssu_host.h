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

// Lets the BULK block-copy kernel use up to `smem_optin` bytes of dynamic shared memory
// (called once per handle by ssu_create, on the handle's device).
cudaError_t copy_prepare(int smem_optin);

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
    unsigned *err = nullptr;  // device: [0] skipped, [1] smallest skipped request, [2] timeouts
    bool has_override = false;
    ssu_launch_t override_launch{};
    bool has_copy_override = false;
    ssu_copy_launch_t copy_override{};
    bool pdl = true;  // launch the VEC and multi-token kernels as programmatic dependents
};
