// Staging of a decode step's per-step operands from page-locked host memory into a dense
// device workspace, for ssu_update_from_host.
//
// A decode step's own inputs are small (batch 128, 16 heads: 332 KB of indices, x, dt, B and
// C against 128 MiB of state traffic), but a copy-engine transfer of them costs a fixed few
// microseconds.  Here every thread of one grid reads one vector of them across the CPU-GPU
// link, so the whole set arrives in about one link round trip, and the update kernel then
// reads them from device memory.  Each operand is a "job": outer x inner rows of row_bytes
// contiguous bytes at byte strides (s_outer, s_inner) in the source, written as dense rows to
// the destination.  The host merges contiguous dimensions into longer rows and picks the
// widest vector (16, 8, 4, 2 or 1 bytes) that the source address, its strides and the row
// length allow.  The destination sections are 256-byte aligned and dense.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ssu_device.cuh"

namespace {

constexpr int kStageJobs = 5;  // indices, x, dt, B, C
constexpr int kStageThreads = 256;

struct StageJob {
    const char *src;
    char *dst;
    long long inner;      // rows per outer index
    long long s_outer;    // source byte stride between outer indices
    long long s_inner;    // source byte stride between inner rows
    long long row_bytes;  // contiguous bytes per row (the destination is dense rows)
    long long cpr;        // vectors per row = row_bytes / vec
    long long chunk0;     // first vector of this job in the grid's vector space
    int vec;              // bytes per vector: 16, 8, 4, 2 or 1
};

struct StageParams {
    StageJob job[kStageJobs];
    int njobs;
    long long total;  // vectors over all jobs
};

template <typename V>
__device__ __forceinline__ void move_vec(const char *s, char *d) {
    *reinterpret_cast<V *>(d) = *reinterpret_cast<const V *>(s);
}

// Byte offsets, in the source and in the destination, of vector `local` of job J.
__host__ __device__ __forceinline__ void stage_offsets(const StageJob &J, long long local,
                                                       long long &src, long long &dst) {
    const long long r = local / J.cpr, k = local - r * J.cpr;
    src = (r / J.inner) * J.s_outer + (r % J.inner) * J.s_inner + k * J.vec;
    dst = r * J.row_bytes + k * J.vec;
}

// One vector per thread and grid-stride iteration.  Waits for the previous grid in the stream
// before the first access (a programmatic dependent launch may start it early) and lets the
// update kernel's CTAs launch once its stores are issued; the update kernel in turn waits for
// this grid to complete, so it sees every staged byte.
__global__ void __launch_bounds__(kStageThreads) ssu_stage_kernel(const StageParams q) {
    pdl_wait();
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; c < q.total;
         c += step) {
        int j = 0;
        while (j + 1 < q.njobs && c >= q.job[j + 1].chunk0) ++j;
        const StageJob &J = q.job[j];
        long long so, dof;
        stage_offsets(J, c - J.chunk0, so, dof);
        const char *s = J.src + so;
        char *d = J.dst + dof;
        switch (J.vec) {
            case 16: move_vec<uint4>(s, d); break;
            case 8: move_vec<uint2>(s, d); break;
            case 4: move_vec<unsigned>(s, d); break;
            case 2: move_vec<unsigned short>(s, d); break;
            default: *d = *s; break;
        }
    }
    pdl_trigger();
}

// Host side: one job from an operand's geometry.  `outer` x `inner` rows of `row_bytes`;
// contiguous dimensions are merged and the vector width chosen from the alignment of the
// source address, its strides and the row length.  `chunk0` is the running vector count.
inline StageJob stage_job(const void *src, void *dst, long long outer, long long inner,
                          long long s_outer, long long s_inner, long long row_bytes,
                          long long &chunk0) {
    if (inner > 1 && s_inner == row_bytes) {
        row_bytes *= inner;
        inner = 1;
        s_inner = 0;
    }
    if (inner == 1 && outer > 1 && s_outer == row_bytes) {
        row_bytes *= outer;
        outer = 1;
        s_outer = 0;
    }
    const unsigned long long addr = reinterpret_cast<unsigned long long>(src);
    int vec = 16;
    while (vec > 1 && (addr % vec != 0 || row_bytes % vec != 0 ||
                       (outer > 1 && s_outer % vec != 0) || (inner > 1 && s_inner % vec != 0)))
        vec >>= 1;
    StageJob j;
    j.src = static_cast<const char *>(src);
    j.dst = static_cast<char *>(dst);
    j.inner = inner;
    j.s_outer = s_outer;
    j.s_inner = s_inner;
    j.row_bytes = row_bytes;
    j.vec = vec;
    j.cpr = row_bytes / vec;
    j.chunk0 = chunk0;
    chunk0 += outer * inner * j.cpr;
    return j;
}

// Launches the staging grid: one vector per thread up to 16 CTAs per SM, grid-stride beyond.
inline cudaError_t launch_stage(const StageParams &q, int sm_count, bool pdl, cudaStream_t st) {
    const long long want = (q.total + kStageThreads - 1) / kStageThreads;
    const long long cap = 16LL * sm_count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
    cfg.blockDim = dim3(kStageThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ssu_stage_kernel, q);
}

}  // namespace
