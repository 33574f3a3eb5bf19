// Multi-token decode step without intermediate states, in chunked matrix form on the tensor
// cores (sm_103a), instantiated by ssu_tokens.cu beside the general kernel of ssu_tokens.cuh.
//
// The step is ssu_tokens.cuh's (T consecutive tokens of every request, vLLM PR #48110, Test
// Plan; each token the Mamba2 decode update of sglang PR #41223, Details):
//   S_t = dA_t S_{t-1} + k_t (x) B_t,   y_t = S_t . C_t + D x_t,   k_t = dt_t x_t (per row).
// Over a chunk of tokens a .. a + len - 1 with Q_t = dA_a ... dA_t, the same recurrence reads
//   S_t = Q_t (S_base + sum_{u<=t} kk_u (x) B_u),           kk_u = k_u / Q_u,
//   y_t = Q_t (S_base . C_t + sum_{u<=t} kk_u G[u][t]) + D x_t,   G[u][t] = B_u . C_t,
// with S_base the state before token a (substitute S_t / Q_t and the step becomes S~_t =
// S~_{t-1} + kk_t B_t).  Per warp of 16 rows that is three small dense contractions: the
// readout S_base [16 x N] . [C_a .. C_{a+7}] [N x 8], the chunk's Gram matrix G [8 x 8] over
// dstate, and the rank-8 update KK [16 x 8] . [B_a .. B_{a+7}]^T [8 x N], all on m16n8k8
// tf32 MMAs with fp32 accumulation.  B and C are bf16, so they are exact in tf32; the fp32
// operands (state, kk, G) are split into a high and a low tf32 part (split_tf32), which
// leaves less than 2^-20 of each value out, so each product keeps close to fp32 accuracy.  The chunk ends before any token whose Q leaves [2^-60, 2^60] (or is not finite);
// a token whose own dA is outside that range takes the plain update alone (elementwise, then
// the same readout).
//
// State layout: the state stays in the MMA accumulator layout from load to store: lane l
// (g = l / 4, i = l % 4) holds rows g and g + 8 of its warp's 16, columns 8j + 2i and
// 8j + 2i + 1 of every 8-column block j.  The readout uses these same registers as its A
// operand by numbering the summation index within each block so that k = i is column 8j + 2i
// and k = i + 4 is column 8j + 2i + 1 (a sum's order of terms is free); B and C are staged
// with the same numbering.
//
// Inputs: each chunk's B, C and x rows are staged into the warp's own shared memory with
// cp.async (16-byte pieces, zero-filled past the last token), together with the tile's state
// loads, so one memory latency covers both.

#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ssu_tokens.cuh"

namespace {

constexpr int kMmaRowsPerWarp = 16;  // the MMA's M
constexpr int kMmaChunk = 8;         // tokens per chunk: the MMA's N (readout) and K (update)
constexpr float kChunkQLo = 0x1p-60f, kChunkQHi = 0x1p60f;

// One warp's staging area: B and C rows of the chunk's tokens (16 bytes of padding per row, so
// that the readout's column-pair loads of 8 tokens hit 32 distinct banks), the warp's 16 rows
// of x per token, and the masked Gram matrix.
template <int N>
struct alignas(16) MmaStage {
    static constexpr int kRow = N + 8;
    unsigned short B[kMmaChunk][kRow];
    unsigned short C[kMmaChunk][kRow];
    unsigned short x[kMmaChunk][kMmaRowsPerWarp];
    float G[kMmaChunk][kMmaChunk];
};

// v = hi + lo + e: hi is v cut to tf32's 10 fraction bits (toward zero), lo the exact rest
// v - hi cut the same way, so |e| < 2^-20 |v|; both are exact tf32 operands.
__device__ __forceinline__ void split_tf32(float f, unsigned &hi, unsigned &lo) {
    constexpr unsigned kMask = 0xffffe000u;
    hi = __float_as_uint(f) & kMask;
    lo = __float_as_uint(f - __uint_as_float(hi)) & kMask;
}

// d += a b for one m16n8k8 tile (tf32 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_tf32(float (&d)[4], unsigned a0, unsigned a1, unsigned a2,
                                         unsigned a3, unsigned b0, unsigned b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes, or zeros where src_bytes = 0 (nothing is read then).
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, int src_bytes) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

// Stage tokens a .. a + 7 (those below T; zeros for the rest) of one warp's chunk.
template <int N>
__device__ __forceinline__ void stage_chunk(const TokenParams &q, MmaStage<N> &st, long long b,
                                            int h, int grp, int row0, int a, int lane) {
    const SsuParams &p = q.p;
    constexpr int kPieces = N / 8;  // 16-byte pieces per token row
    const unsigned short *Bb =
        reinterpret_cast<const unsigned short *>(p.B) + b * p.B_b + grp * p.B_g;
    const unsigned short *Cb =
        reinterpret_cast<const unsigned short *>(p.C) + b * p.C_b + grp * p.C_g;
#pragma unroll
    for (int i = 0; i < (2 * kMmaChunk * kPieces) / 32; ++i) {
        const int idx = i * 32 + lane;
        const bool isC = idx >= kMmaChunk * kPieces;
        const int rem = isC ? idx - kMmaChunk * kPieces : idx;
        const int tok = rem / kPieces, piece = rem % kPieces;
        const bool live = a + tok < q.tokens;
        const unsigned short *src =
            (isC ? Cb + (live ? (a + tok) * q.C_t : 0) : Bb + (live ? (a + tok) * q.B_t : 0)) +
            piece * 8;
        unsigned short *dst = (isC ? st.C[tok] : st.B[tok]) + piece * 8;
        cp_async16_zfill(dst, src, live ? 16 : 0);
    }
    if (lane < 2 * kMmaChunk) {
        const int tok = lane >> 1, half = lane & 1;
        const bool live = a + tok < q.tokens && row0 + 8 * half < p.headdim;
        const unsigned short *src = reinterpret_cast<const unsigned short *>(p.x) + b * p.x_b +
                                    h * p.x_h + (live ? (a + tok) * q.x_t + row0 + 8 * half : 0);
        cp_async16_zfill(&st.x[tok][8 * half], src, live ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// A warp's tile: 16 rows (row0 ..) of one head of one request.
struct MmaTile {
    long long b;
    int h, row0;
};

// The chunks of one tile: S holds the tile's state (accumulator layout) on entry and the state
// after its T tokens on return.  Chunk 0's copies are issued (not waited for); dt_raw holds,
// in lanes 0..7, the bf16 dt bits of tokens 0..7.
template <int N>
__device__ __forceinline__ void mma_tile_tokens(const TokenParams &q, MmaStage<N> &st,
                                                float (&S)[N / 8][4], const MmaTile &tl,
                                                unsigned short dt_raw, int lane) {
    constexpr int NT = N / 8;
    const SsuParams &p = q.p;
    const int g = lane >> 2, i4 = lane & 3;
    const long long b = tl.b;
    const int h = tl.h, row0 = tl.row0;
    const bool liveA = row0 + g < p.headdim, liveB = row0 + g + 8 < p.headdim;
    const int grp = group_of(h, p.group_magic);
    const float bias = p.dt_bias[h * p.bias_h];
    const float Ah = p.A[h * p.A_h];
    const float Dh = p.D[h * p.D_h];
    for (int a = 0; a < q.tokens;) {
        // This chunk's scalars, token a + j in lane j < 8: dt, dA and the running product.
        const int u = a + (lane & 7);
        float dtv = 0.f, dA = 1.f;
        if (lane < kMmaChunk && u < q.tokens) {
            const unsigned short raw =
                a == 0 ? dt_raw
                       : reinterpret_cast<const unsigned short *>(
                             p.dt)[b * p.dt_b + u * q.dt_t + h * p.dt_h];
            dtv = softplus_f32(widen_bf16(raw) + bias);
            dA = expf(dtv * Ah);
        }
        float Q = dA;
#pragma unroll
        for (int d = 1; d < kMmaChunk; d <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, Q, d);
            if ((lane & 7) >= d) Q = o * Q;
        }
        const int cnt = min(kMmaChunk, q.tokens - a);
        const bool in_range = Q >= kChunkQLo && Q <= kChunkQHi;
        const unsigned bad = __ballot_sync(0xffffffffu, lane < cnt && !in_range);
        const int lead = bad ? __ffs(bad) - 1 : cnt;  // leading tokens in range
        const bool plain = lead == 0;
        const int len = plain ? 1 : lead;
        const float kq = plain ? dtv : __fdiv_rn(dtv, Q);
        // The chunk's staged inputs are needed from here on (their copies ran meanwhile).
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();  // every lane's pieces of the chunk are visible to all
        const float kq0 = __shfl_sync(0xffffffffu, kq, i4);
        const float kq1 = __shfl_sync(0xffffffffu, kq, i4 + 4);
        if (plain) {
            // Token a alone, plain update S = S dA + k B, elementwise (the warp takes this
            // branch as one: `plain` comes from a ballot).
            const float dA0 = __shfl_sync(0xffffffffu, dA, 0);
            const float dt0 = __shfl_sync(0xffffffffu, dtv, 0);
            const float k0 = dt0 * widen_bf16(st.x[0][g]);
            const float k1 = dt0 * widen_bf16(st.x[0][g + 8]);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const unsigned w = *reinterpret_cast<const unsigned *>(&st.B[0][8 * j + 2 * i4]);
                const float b0 = bf16_lo(w), b1 = bf16_hi(w);
                S[j][0] = fmaf(S[j][0], dA0, k0 * b0);
                S[j][1] = fmaf(S[j][1], dA0, k0 * b1);
                S[j][2] = fmaf(S[j][2], dA0, k1 * b0);
                S[j][3] = fmaf(S[j][3], dA0, k1 * b1);
            }
        }
        // KK (A operand of the correction and of the update): rows g / g + 8, tokens i4 and
        // i4 + 4 of the chunk; zero past the chunk and in a plain chunk.
        unsigned kh[4], kl[4];
        {
            const bool u0 = !plain && i4 < len, u1 = !plain && i4 + 4 < len;
            const float kk[4] = {u0 ? kq0 * widen_bf16(st.x[i4][g]) : 0.f,
                                 u0 ? kq0 * widen_bf16(st.x[i4][g + 8]) : 0.f,
                                 u1 ? kq1 * widen_bf16(st.x[i4 + 4][g]) : 0.f,
                                 u1 ? kq1 * widen_bf16(st.x[i4 + 4][g + 8]) : 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e) split_tf32(kk[e], kh[e], kl[e]);
        }
        // Readout S_base . C_t and the Gram matrix B_u . C_t, block by block (four readout and
        // two Gram accumulators, so that the MMAs of consecutive blocks do not wait on each
        // other; summed at the end).
        float Yp[4][4] = {}, Gp[2][4] = {};
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const unsigned cw = *reinterpret_cast<const unsigned *>(&st.C[g][8 * j + 2 * i4]);
            const unsigned bw = *reinterpret_cast<const unsigned *>(&st.B[g][8 * j + 2 * i4]);
            const unsigned c0 = __float_as_uint(bf16_lo(cw)), c1 = __float_as_uint(bf16_hi(cw));
            mma_tf32(Gp[j & 1], __float_as_uint(bf16_lo(bw)), 0u, __float_as_uint(bf16_hi(bw)),
                     0u, c0, c1);
            unsigned h0, l0, h1, l1, h2, l2, h3, l3;
            split_tf32(S[j][0], h0, l0);  // (row g, k = i4)
            split_tf32(S[j][2], h1, l1);  // (row g + 8, k = i4)
            split_tf32(S[j][1], h2, l2);  // (row g, k = i4 + 4)
            split_tf32(S[j][3], h3, l3);  // (row g + 8, k = i4 + 4)
            mma_tf32(Yp[2 * (j & 1)], h0, h1, h2, h3, c0, c1);
            mma_tf32(Yp[2 * (j & 1) + 1], l0, l1, l2, l3, c0, c1);
        }
        float Y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) Y[e] = (Yp[0][e] + Yp[2][e]) + (Yp[1][e] + Yp[3][e]);
        // The Gram matrix masked to u <= t < len, through shared memory to the layout of the
        // correction's B operand (k = u, n = t).
        {
            const int t0 = 2 * i4, t1 = 2 * i4 + 1;
            st.G[g][t0] = (g <= t0 && t0 < len) ? Gp[0][0] + Gp[1][0] : 0.f;
            st.G[g][t1] = (g <= t1 && t1 < len) ? Gp[0][1] + Gp[1][1] : 0.f;
        }
        __syncwarp();
        if (!plain) {
            unsigned gh0, gl0, gh1, gl1;
            split_tf32(st.G[i4][g], gh0, gl0);
            split_tf32(st.G[i4 + 4][g], gh1, gl1);
            mma_tf32(Y, kh[0], kh[1], kh[2], kh[3], gh0, gh1);
            mma_tf32(Y, kh[0], kh[1], kh[2], kh[3], gl0, gl1);
            mma_tf32(Y, kl[0], kl[1], kl[2], kl[3], gh0, gh1);
        }
        // Readouts: Y[0] (row g, t = 2 i4), Y[1] (g, 2 i4 + 1), Y[2] (g + 8, 2 i4), Y[3].
        {
            const float q0 = __shfl_sync(0xffffffffu, Q, 2 * i4);
            const float q1 = __shfl_sync(0xffffffffu, Q, 2 * i4 + 1);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 2 * i4 + (e & 1);
                const int r = e < 2 ? g : g + 8;
                const bool live = t < len && (e < 2 ? liveA : liveB);
                const float rs = plain ? 1.f : ((e & 1) ? q1 : q0);
                if (live) {
                    const float xv = widen_bf16(st.x[t][r]);
                    p.out[b * p.out_b + (a + t) * q.out_t + h * p.out_h + row0 + r] =
                        __float2bfloat16_rn(fmaf(Dh, xv, rs * Y[e]));
                }
            }
        }
        if (!plain) {
            // S_base + KK B^T, then back to the state's own scale (times Q of the last).
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const unsigned b0 = __float_as_uint(widen_bf16(st.B[i4][8 * j + g]));
                const unsigned b1 = __float_as_uint(widen_bf16(st.B[i4 + 4][8 * j + g]));
                mma_tf32(S[j], kh[0], kh[1], kh[2], kh[3], b0, b1);
                mma_tf32(S[j], kl[0], kl[1], kl[2], kl[3], b0, b1);
            }
            const float ql = __shfl_sync(0xffffffffu, Q, len - 1);
            const float2 q2 = make_float2(ql, ql);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const float2 s0 = __fmul2_rn(make_float2(S[j][0], S[j][1]), q2);
                const float2 s1 = __fmul2_rn(make_float2(S[j][2], S[j][3]), q2);
                S[j][0] = s0.x, S[j][1] = s0.y, S[j][2] = s1.x, S[j][3] = s1.y;
            }
        }
        a += len;
        if (a < q.tokens) {
            __syncwarp();  // every lane is done with this chunk's staging area
            stage_chunk<N>(q, st, b, h, grp, row0, a, lane);
        }
    }
}

constexpr int kMmaWarpsPerCta = 4;  // 64 rows per CTA
constexpr int kMmaCtasPerSm = 4;    // 16 warps: at most 128 registers a thread

// One CTA per (slab of 64 rows, head, request); warp w takes rows 16w .. 16w + 15 of the slab.
// Each warp loads its tile's state straight into registers (accumulator layout) and stages its
// first chunk of inputs at the same time, so that one memory latency covers both.
template <int N, typename ST, bool kIdx64>
__global__ void __launch_bounds__(32 * kMmaWarpsPerCta, kMmaCtasPerSm)
    ssu_tokens_mma_kernel(const __grid_constant__ TokenParams q) {
    constexpr int NT = N / 8;
    __shared__ MmaStage<N> stage[kMmaWarpsPerCta];
    pdl_wait();
    const SsuParams &p = q.p;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2, i4 = lane & 3;
    MmaStage<N> &st = stage[warp];
    MmaTile tl;
    tl.h = blockIdx.y;
    tl.row0 = (blockIdx.x * (blockDim.x >> 5) + warp) * kMmaRowsPerWarp;  // (the launch's width)
    if (tl.row0 < p.headdim) {
        const int rA = tl.row0 + g;
        const bool liveA = rA < p.headdim, liveB = rA + 8 < p.headdim;
        const int grp = group_of(tl.h, p.group_magic);
        for (long long b = blockIdx.z; b < p.batch; b += gridDim.z) {
            tl.b = b;
            const long long s = load_slot<kIdx64>(p, b);
            if (s < 0 || s >= p.pool_size) {
                if (tl.h == 0 && blockIdx.x == 0 && threadIdx.x == 0) record_skip(p, b);
                continue;
            }
            ST *sA = static_cast<ST *>(p.state) + s * p.st_pool + tl.h * p.st_head +
                     rA * p.st_row + 2 * i4;
            ST *sB = sA + 8 * p.st_row;
            // S[j] = (row g, 8j+2i), (g, 8j+2i+1), (g+8, 8j+2i), (g+8, 8j+2i+1)
            float S[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (sizeof(ST) == 4) {
                    const float2 va = liveA ? __ldcs(reinterpret_cast<const float2 *>(sA + 8 * j))
                                            : make_float2(0.f, 0.f);
                    const float2 vb = liveB ? __ldcs(reinterpret_cast<const float2 *>(sB + 8 * j))
                                            : make_float2(0.f, 0.f);
                    S[j][0] = va.x, S[j][1] = va.y, S[j][2] = vb.x, S[j][3] = vb.y;
                } else {
                    const unsigned wa =
                        liveA ? __ldcs(reinterpret_cast<const unsigned *>(sA + 8 * j)) : 0u;
                    const unsigned wb =
                        liveB ? __ldcs(reinterpret_cast<const unsigned *>(sB + 8 * j)) : 0u;
                    S[j][0] = bf16_lo(wa), S[j][1] = bf16_hi(wa);
                    S[j][2] = bf16_lo(wb), S[j][3] = bf16_hi(wb);
                }
            }
            const unsigned short dt_raw =
                lane < kMmaChunk && lane < q.tokens
                    ? reinterpret_cast<const unsigned short *>(
                          p.dt)[b * p.dt_b + lane * q.dt_t + tl.h * p.dt_h]
                    : static_cast<unsigned short>(0);
            __syncwarp();  // the previous request's reads of the staging area are done
            stage_chunk<N>(q, st, b, tl.h, grp, tl.row0, 0, lane);
            mma_tile_tokens<N>(q, st, S, tl, dt_raw, lane);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (sizeof(ST) == 4) {
                    if (liveA)
                        __stcs(reinterpret_cast<float2 *>(sA + 8 * j),
                               make_float2(S[j][0], S[j][1]));
                    if (liveB)
                        __stcs(reinterpret_cast<float2 *>(sB + 8 * j),
                               make_float2(S[j][2], S[j][3]));
                } else {
                    if (liveA)
                        __stcs(reinterpret_cast<unsigned *>(sA + 8 * j),
                               f2_to_bf2(S[j][0], S[j][1]));
                    if (liveB)
                        __stcs(reinterpret_cast<unsigned *>(sB + 8 * j),
                               f2_to_bf2(S[j][2], S[j][3]));
                }
            }
        }
    }
    pdl_trigger();
}

template <int N, typename ST, bool kIdx64>
cudaError_t launch_tokens_mma(const TokenParams &q, dim3 grid, int warps, bool pdl,
                              cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * warps);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ssu_tokens_mma_kernel<N, ST, kIdx64>, q);
}

}  // namespace
