// Multi-token decode-step kernels with a prefetch ring of 4 tokens (used from 3 tokens per
// call on, up to dstate 128), compiled apart from ssu_tokens.cu so the two sets of
// instantiations build in parallel.

#include <cstring>

#include "ssu_host.h"
#include "ssu_tokens.cuh"

namespace ssu_host {

cudaError_t tokens_launch_depth4(const void *params, size_t bytes, int nc, bool bf16, bool i64,
                                 int rpw, int wpc, dim3 grid, bool pdl, cudaStream_t st) {
    TokenParams q;
    if (bytes != sizeof(q)) return cudaErrorInvalidValue;
    std::memcpy(&q, params, sizeof(q));
    return launch_tokens_depth<4>(q, nc, bf16, i64, rpw, wpc, grid, pdl, st);
}

}  // namespace ssu_host
