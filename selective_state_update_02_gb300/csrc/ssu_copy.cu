// State-block copy for GB300 (sm_103a): block src_idx[i] -> block dst_idx[i] of every state
// tensor (vLLM PR #48110, Purpose and Test Plan / Microbenchmark describe the operation: the
// temporal and conv states of each hybrid layer are copied between cache blocks under prefix
// caching and multi-token speculation).  Pure data movement, bound by HBM bandwidth.
//
// Work decomposition.  Every (tensor, request) block is cut into chunks of `chunk_bytes`;
// chunks of tensor t occupy a contiguous range of a global chunk index (tensor-major, then
// request, then chunk), so the whole call is one flat list that persistent CTAs stride through.
//
// Each thread moves `vectors` 16-byte words per pass, all loads issued before the stores.
// (A variant driving the TMA engine's 1-D bulk copies through a shared-memory ring was measured
// slower at every size and is not part of the library.)

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ssu.h"
#include "ssu_device.cuh"
#include "ssu_host.h"

using ssu_host::aligned;
using ssu_host::DeviceGuard;
using ssu_host::fail;
using ssu_host::ok;

namespace {

struct CopyTensor {
    char *base;
    long long block_bytes;
    long long stride;
    long long num_blocks;
    long long chunks;       // chunks per block
    long long chunk_begin;  // first global chunk index of this tensor
};

struct CopyParams {
    CopyTensor t[SSU_COPY_MAX_TENSORS];
    const void *src;
    const void *dst;
    long long n;
    long long total_chunks;
    long long chunk_bytes;
    int num_tensors;
    int idx64;
    unsigned *err;  // [0] skipped requests, [1] smallest skipped request
};

struct ChunkRef {
    const char *src;
    char *dst;
    unsigned bytes;
    bool valid;
};

__device__ __forceinline__ long long load_id(const void *ids, int idx64, long long i) {
    return idx64 ? __ldg(static_cast<const long long *>(ids) + i)
                 : static_cast<long long>(__ldg(static_cast<const int *>(ids) + i));
}

// Locates global chunk c: its tensor, request, source and destination.
__device__ __forceinline__ ChunkRef locate_chunk(const CopyParams &p, long long c) {
    int t = 0;
    while (t + 1 < p.num_tensors && c >= p.t[t + 1].chunk_begin) ++t;
    const CopyTensor &T = p.t[t];
    const long long local = c - T.chunk_begin;
    const long long i = local / T.chunks;
    const long long k = local - i * T.chunks;
    const long long s = load_id(p.src, p.idx64, i);
    const long long d = load_id(p.dst, p.idx64, i);
    ChunkRef r;
    // A request is skipped for every tensor if any of its ids is out of any tensor's range.
    bool valid = true;
    for (int u = 0; u < p.num_tensors; ++u)
        valid = valid && s >= 0 && d >= 0 && s < p.t[u].num_blocks && d < p.t[u].num_blocks;
    r.valid = valid;
    const long long off = k * p.chunk_bytes;
    const long long rest = T.block_bytes - off;
    r.bytes = static_cast<unsigned>(rest < p.chunk_bytes ? rest : p.chunk_bytes);
    r.src = T.base + s * T.stride + off;
    r.dst = T.base + d * T.stride + off;
    if (!valid && t == 0 && k == 0 && (threadIdx.x == 0)) {
        atomicAdd(&p.err[0], 1u);
        atomicMin(&p.err[1], static_cast<unsigned>(i));
    }
    return r;
}

// Launched as a programmatic dependent when the handle says so: nothing is read or written
// before the previous kernel in the stream has completed (pdl_wait), and each CTA lets a
// dependent launch start once its last stores are issued.
template <int V>
__global__ void __launch_bounds__(256) copy_vec_kernel(const __grid_constant__ CopyParams p) {
    pdl_wait();
    const long long pass = static_cast<long long>(blockDim.x) * 16 * V;
    for (long long c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
        const ChunkRef r = locate_chunk(p, c);
        if (!r.valid) continue;
        for (long long base = 0; base < r.bytes; base += pass) {
            uint4 v[V];
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const long long o = base + (static_cast<long long>(u) * blockDim.x + threadIdx.x) * 16;
                if (o < r.bytes) v[u] = __ldcs(reinterpret_cast<const uint4 *>(r.src + o));
            }
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const long long o = base + (static_cast<long long>(u) * blockDim.x + threadIdx.x) * 16;
                if (o < r.bytes) __stcs(reinterpret_cast<uint4 *>(r.dst + o), v[u]);
            }
        }
    }
    pdl_trigger();
}

template <int V>
cudaError_t launch_copy_vec_one(const CopyParams &p, int threads, unsigned grid, bool pdl,
                                cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, copy_vec_kernel<V>, p);
}

cudaError_t launch_copy_vec(const CopyParams &p, int vectors, int threads, unsigned grid,
                            bool pdl, cudaStream_t st) {
    switch (vectors) {
        case 1: return launch_copy_vec_one<1>(p, threads, grid, pdl, st);
        case 2: return launch_copy_vec_one<2>(p, threads, grid, pdl, st);
        case 4: return launch_copy_vec_one<4>(p, threads, grid, pdl, st);
        case 8: return launch_copy_vec_one<8>(p, threads, grid, pdl, st);
        case 16: return launch_copy_vec_one<16>(p, threads, grid, pdl, st);
        default: return cudaErrorInvalidValue;
    }
}

using VecCopyKernel = void (*)(CopyParams);

VecCopyKernel vec_copy_kernel(int vectors) {
    switch (vectors) {
        case 1: return copy_vec_kernel<1>;
        case 2: return copy_vec_kernel<2>;
        case 4: return copy_vec_kernel<4>;
        case 8: return copy_vec_kernel<8>;
        case 16: return copy_vec_kernel<16>;
        default: return nullptr;
    }
}

bool copy_launch_ok(const ssu_copy_launch_t &l) {
    const int c = l.chunk_kib;
    if (c != 4 && c != 8 && c != 16 && c != 32 && c != 64) return false;
    if (l.mode == SSU_COPY_VEC)
        return vec_copy_kernel(l.stages) != nullptr && l.threads >= 32 && l.threads <= 256 &&
               l.threads % 32 == 0;
    return false;
}

// Built-in choice, from the cold-L2 sweep on GB300 (bench.py --copy --sweep): 128-thread VEC
// CTAs; calls under 1 GiB use 16 KiB chunks with 8 x 16 bytes per thread per pass, larger
// calls 64 KiB chunks with 16 x 16 bytes (one pass per chunk either way).
ssu_copy_launch_t copy_table(long long total_bytes) {
    if (total_bytes >= (1LL << 30)) return ssu_copy_launch_t{SSU_COPY_VEC, 64, 16, 128};
    return ssu_copy_launch_t{SSU_COPY_VEC, 16, 8, 128};
}

}  // namespace

extern "C" {

ssu_status_t ssu_copy_set_launch(ssu_handle_t handle, const ssu_copy_launch_t *launch) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    if (!launch || launch->mode == SSU_COPY_AUTO) {
        handle->has_copy_override = false;
        return ok();
    }
    if (!copy_launch_ok(*launch))
        return fail(SSU_ERR_UNSUPPORTED, "copy launch mode=%d chunk_kib=%d stages=%d threads=%d",
                    launch->mode, launch->chunk_kib, launch->stages, launch->threads);
    handle->copy_override = *launch;
    handle->has_copy_override = true;
    return ok();
}

ssu_status_t ssu_copy_blocks(ssu_handle_t handle, const ssu_block_tensor_t *tensors,
                             int32_t num_tensors, const void *src_idx, const void *dst_idx,
                             int64_t n, int32_t index_dtype, ssu_stream_t stream) {
    if (!handle) return fail(SSU_ERR_INVALID_ARG, "NULL handle");
    if (n < 0) return fail(SSU_ERR_INVALID_ARG, "n < 0");
    if (num_tensors < 1 || num_tensors > SSU_COPY_MAX_TENSORS)
        return fail(SSU_ERR_INVALID_ARG, "num_tensors %d outside 1..%d", num_tensors,
                    SSU_COPY_MAX_TENSORS);
    if (!tensors) return fail(SSU_ERR_INVALID_ARG, "tensors is NULL");
    if (index_dtype != SSU_INDEX_I32 && index_dtype != SSU_INDEX_I64)
        return fail(SSU_ERR_INVALID_ARG, "index_dtype %d is neither I32 nor I64", index_dtype);
    for (int t = 0; t < num_tensors; ++t) {
        const ssu_block_tensor_t &T = tensors[t];
        if (!T.base) return fail(SSU_ERR_INVALID_ARG, "tensor %d: NULL base", t);
        if (T.block_bytes <= 0 || T.num_blocks < 0 || T.block_stride_bytes < T.block_bytes)
            return fail(SSU_ERR_INVALID_ARG, "tensor %d: bad block size/stride/count", t);
        if (!aligned(T.base, 16) || T.block_bytes % 16 || T.block_stride_bytes % 16)
            return fail(SSU_ERR_MISALIGNED,
                        "tensor %d: base, block size and stride must be multiples of 16 bytes",
                        t);
    }
    if (n == 0) return ok();
    if (!src_idx || !dst_idx) return fail(SSU_ERR_INVALID_ARG, "src_idx or dst_idx is NULL");
    const unsigned isz = index_dtype == SSU_INDEX_I64 ? 8 : 4;
    if (!aligned(src_idx, isz) || !aligned(dst_idx, isz))
        return fail(SSU_ERR_MISALIGNED, "index arrays are not aligned to their type");
    if (n > UINT_MAX - 1) return fail(SSU_ERR_UNSUPPORTED, "n exceeds 2^32 - 2");

    long long total_bytes = 0;
    for (int t = 0; t < num_tensors; ++t) total_bytes += n * tensors[t].block_bytes;
    const ssu_copy_launch_t l =
        handle->has_copy_override ? handle->copy_override : copy_table(total_bytes);
    CopyParams p{};
    p.chunk_bytes = static_cast<long long>(l.chunk_kib) * 1024;
    long long chunks = 0;
    for (int t = 0; t < num_tensors; ++t) {
        CopyTensor &T = p.t[t];
        T.base = static_cast<char *>(tensors[t].base);
        T.block_bytes = tensors[t].block_bytes;
        T.stride = tensors[t].block_stride_bytes;
        T.num_blocks = tensors[t].num_blocks;
        T.chunks = (T.block_bytes + p.chunk_bytes - 1) / p.chunk_bytes;
        T.chunk_begin = chunks;
        chunks += n * T.chunks;
    }
    p.src = src_idx;
    p.dst = dst_idx;
    p.n = n;
    p.total_chunks = chunks;
    p.num_tensors = num_tensors;
    p.idx64 = index_dtype == SSU_INDEX_I64;
    p.err = handle->err;

    DeviceGuard guard(handle->device);
    if (guard.err != cudaSuccess)
        return fail(SSU_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(guard.err));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vec_copy_kernel(l.stages),
                                                      l.threads, 0);
    if (e == cudaSuccess && per_sm < 1) e = cudaErrorInvalidConfiguration;
    if (e == cudaSuccess) {
        const long long slots = static_cast<long long>(per_sm) * handle->sm_count;
        const unsigned grid = static_cast<unsigned>(chunks < slots ? chunks : slots);
        e = launch_copy_vec(p, l.stages, l.threads, grid, handle->pdl, cs);
    }
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "copy launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"
