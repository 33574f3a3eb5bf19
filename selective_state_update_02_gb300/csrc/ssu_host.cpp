// Host-side helpers of libssu: error messages, argument validation, status names.

#include <climits>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <vector>

#include "ssu_host.h"

namespace ssu_host {


namespace {
thread_local std::string g_last_error;
}  // namespace

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

ssu_status_t validate_impl(const void *state_pool, const void *idx, const uint16_t *x,
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
    if (s.state_dtype != SSU_STATE_F32 && s.state_dtype != SSU_STATE_BF16)
        return fail(SSU_ERR_INVALID_ARG, "state_dtype %d is neither F32 nor BF16", s.state_dtype);
    if (s.dstate != 64 && s.dstate != 128 && s.dstate != 256)
        return fail(SSU_ERR_UNSUPPORTED, "dstate %lld: this build implements 64, 128 and 256",
                    (long long)s.dstate);
    if (s.headdim > (1 << 20) || s.nheads > 65535)
        return fail(SSU_ERR_UNSUPPORTED, "headdim is limited to 2^20 and nheads to 65535");
    if (s.batch == 0) return ok();  // nothing is read or written: strides are irrelevant

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
    const int per16 = s.state_dtype == SSU_STATE_BF16 ? 8 : 4;  // elements per 16 bytes
    for (int j = 0; j < 3; ++j)
        if (st->state[j] % per16 != 0)
            return fail(SSU_ERR_MISALIGNED,
                        "state stride %d (%lld elements) is not a multiple of 16 bytes", j,
                        (long long)st->state[j]);

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

int rows_per_instruction(int64_t dstate, int32_t state_dtype) {
    const int64_t row_bytes = dstate * (state_dtype == SSU_STATE_BF16 ? 2 : 4);
    return row_bytes >= 512 ? 1 : static_cast<int>(512 / row_bytes);
}

bool rows_per_warp_ok(int rows_per_warp, int64_t dstate, int32_t state_dtype) {
    if (dstate == 128 && state_dtype == SSU_STATE_F32 && rows_per_warp == 16) return true;
    const int rpi = rows_per_instruction(dstate, state_dtype);
    for (int slots = 1; slots <= 8; slots *= 2)
        if (rows_per_warp == slots * rpi) return true;
    return false;
}

}  // namespace ssu_host

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

const char *ssu_last_error(void) { return ssu_host::g_last_error.c_str(); }

ssu_status_t ssu_check_indices(const void *host_indices, int64_t n, int32_t index_dtype,
                               int64_t pool_size, int64_t *first_bad) {
    using ssu_host::fail;
    if (first_bad) *first_bad = -1;
    if (n < 0 || pool_size < 0) return fail(SSU_ERR_INVALID_ARG, "n and pool_size must be >= 0");
    if (index_dtype != SSU_INDEX_I32 && index_dtype != SSU_INDEX_I64)
        return fail(SSU_ERR_INVALID_ARG, "index_dtype %d is neither I32 nor I64", index_dtype);
    if (n == 0) return ssu_host::ok();
    if (!host_indices) return fail(SSU_ERR_INVALID_ARG, "host_indices is NULL");
    // One bit per slot marks the slots seen so far.
    std::vector<unsigned char> seen(static_cast<size_t>((pool_size + 7) / 8), 0);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t s = index_dtype == SSU_INDEX_I64
                              ? static_cast<const int64_t *>(host_indices)[i]
                              : static_cast<int64_t>(static_cast<const int32_t *>(host_indices)[i]);
        if (s < 0 || s >= pool_size) {
            if (first_bad) *first_bad = i;
            return fail(SSU_ERR_INVALID_ARG, "request %lld names slot %lld outside [0, %lld)",
                        (long long)i, (long long)s, (long long)pool_size);
        }
        unsigned char &byte = seen[static_cast<size_t>(s >> 3)];
        const unsigned char bit = static_cast<unsigned char>(1u << (s & 7));
        if (byte & bit) {
            if (first_bad) *first_bad = i;
            return fail(SSU_ERR_INVALID_ARG, "request %lld repeats slot %lld", (long long)i,
                        (long long)s);
        }
        byte |= bit;
    }
    return ssu_host::ok();
}

}  // extern "C"
