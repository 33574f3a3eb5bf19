// BULK kernel of the decode step (fp32 state, dstate 128).  Persistent CTAs (as many as fit on
// the SMs) stream tiles of `tile_rows` rows through a ring of shared-memory stages.  Warp 0 is
// the producer: it reads the slot index of each tile ahead of time and issues a bulk
// asynchronous copy (the TMA engine's 1-D `cp.async.bulk`) of the tile's contiguous rows into a
// free stage, completion counted on the stage's mbarrier.  The compute warps read their rows
// out of the stage into registers, hand the stage back at once (the producer refills it while
// they work), update the rows, store them in place with 16-byte vector stores and write the
// readout.  Loads in flight are bounded by shared memory (stages x tile), not by registers.
// Every mbarrier wait is bounded in time; a timeout raises an error counter and the CTA stops
// after its copies in flight have landed.
#pragma once

#include "ssu_device.cuh"

namespace {

// Shared-memory layout of the BULK kernel: barriers and per-stage slots, then the stages.
struct BulkSmem {
    uint64_t *full;   // [stages] producer -> compute: stage loaded (or its tile skipped)
    uint64_t *freed;  // [stages] compute -> producer: every compute warp has read the stage
    long long *slot;  // [stages] slot of the tile in the stage, -1 when skipped
    float *buf;       // [stages][tile_rows][128]
};

__host__ __device__ constexpr unsigned bulk_header_bytes(int stages) {
    return ((static_cast<unsigned>(stages) * 24u + 127u) / 128u) * 128u;
}

__device__ __forceinline__ BulkSmem bulk_smem(unsigned char *base, int stages) {
    BulkSmem s;
    s.full = reinterpret_cast<uint64_t *>(base);
    s.freed = s.full + stages;
    s.slot = reinterpret_cast<long long *>(s.freed + stages);
    s.buf = reinterpret_cast<float *>(base + bulk_header_bytes(stages));
    return s;
}

// Coordinates of global tile t.
struct TileCoord {
    long long b;
    int h, row0, rows;
};

__device__ __forceinline__ TileCoord tile_coord(const SsuParams &p, long long t) {
    TileCoord c;  // t < 2^31 (checked on the host), so 32-bit division suffices
    const unsigned tt = static_cast<unsigned>(t);
    const unsigned unit = tt / static_cast<unsigned>(p.slabs);
    const int slab = static_cast<int>(tt - unit * static_cast<unsigned>(p.slabs));
    c.h = static_cast<int>(unit % static_cast<unsigned>(p.nheads));
    c.b = static_cast<long long>(unit / static_cast<unsigned>(p.nheads));
    c.row0 = slab * p.rows_per_cta;
    c.rows = min(p.rows_per_cta, p.headdim - c.row0);
    return c;
}

// Per-tile inputs of one compute warp, loaded one tile ahead of their use.
struct TileInputs {
    float dt, bias, A, D;
    float bb[4], cc[4];
    float x;  // lane r < RPW: x of this warp's row r of the tile
};

template <int RPW>
__device__ __forceinline__ TileInputs load_tile_inputs(const SsuParams &p, const TileCoord &c,
                                                       int cw, int lane) {
    TileInputs in;
    const long long b = c.b;
    const int h = c.h;
    in.dt = __bfloat162float(p.dt[b * p.dt_b + h * p.dt_h]);
    in.bias = p.dt_bias[h * p.bias_h];
    in.A = p.A[h * p.A_h];
    in.D = p.D[h * p.D_h];
    const int g = h / p.heads_per_group;
    const __nv_bfloat16 *Bp = p.B + b * p.B_b + g * p.B_g + lane * 4;
    const __nv_bfloat16 *Cp = p.C + b * p.C_b + g * p.C_g + lane * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        in.bb[j] = __bfloat162float(Bp[j]);
        in.cc[j] = __bfloat162float(Cp[j]);
    }
    const int row = cw * RPW + lane;
    in.x = (lane < RPW && row < c.rows)
               ? __bfloat162float(p.x[b * p.x_b + h * p.x_h + c.row0 + row])
               : 0.f;
    return in;
}

// Producer warp 0 issues the bulk loads; compute warps 1..W update rows and store them from
// registers.  A stage is handed back to the producer as soon as every compute warp has read
// its rows out of it, so the producer refills it while the update and the stores proceed.
template <int RPW, bool kIdx64>
__global__ void __launch_bounds__(32 * (1 + kMaxBulkWarps))
    ssu_bulk_kernel(const __grid_constant__ SsuParams p, const BulkShape q) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int stages = q.stages;
    const BulkSmem sm = bulk_smem(smem_raw, stages);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int compute_warps = static_cast<int>(blockDim.x >> 5) - 1;
    const long long G = gridDim.x;
    const long long cta = blockIdx.x;
    const long long n_my = (q.tiles - cta + G - 1) / G;  // tiles cta, cta + G, ...
    constexpr int kRowFloats = kDstate;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.freed[s], static_cast<unsigned>(32 * compute_warps));
        }
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------- producer warp ----------------
        // Slots of this CTA's tiles in windows of 32 (lane l holds tile win + l); the next
        // window is loaded one window ahead.
        auto slot_of_tile = [&](long long i) -> long long {
            if (i >= n_my) return -1;
            const TileCoord c = tile_coord(p, cta + i * G);
            return load_slot<kIdx64>(p, c.b);
        };
        long long win = 0;
        long long win_cur = slot_of_tile(lane);
        long long win_next = slot_of_tile(32 + lane);
        auto issue_load = [&](long long j) {
            if (j >= win + 32) {  // j advances by one per call
                win += 32;
                win_cur = win_next;
                win_next = slot_of_tile(win + 32 + lane);
            }
            const long long s = __shfl_sync(0xffffffffu, win_cur, static_cast<int>(j - win));
            const int st = static_cast<int>(j % stages);
            const TileCoord c = tile_coord(p, cta + j * G);
            const bool valid = s >= 0 && s < p.pool_size;
            if (lane == 0) {
                sm.slot[st] = valid ? s : -1;
                if (valid) {
                    const unsigned bytes = static_cast<unsigned>(c.rows) * kRowBytes;
                    mbar_arrive_expect_tx(&sm.full[st], bytes);
                    bulk_load(sm.buf + static_cast<size_t>(st) * p.rows_per_cta * kRowFloats,
                              static_cast<float *>(p.state) + s * p.st_pool + c.h * p.st_head + c.row0 * p.st_row,
                              bytes, &sm.full[st]);
                } else {
                    if (c.h == 0 && c.row0 == 0) record_skip(p, c.b);
                    mbar_arrive(&sm.full[st]);
                }
            }
            __syncwarp();
        };
        const long long first = n_my < stages ? n_my : stages;
        for (long long j = 0; j < first; ++j) issue_load(j);
        long long issued = first;
        bool failed = false;
        for (long long i = 0; i + stages < n_my; ++i) {
            const int st = static_cast<int>(i % stages);
            const bool ok = mbar_wait(&sm.freed[st], static_cast<unsigned>((i / stages) & 1));
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                break;
            }
            issue_load(i + stages);
            issued = i + stages + 1;
        }
        if (failed && lane == 0) {
            atomicAdd(&p.err[2], 1u);
            // Loads in flight must land before the CTA's shared memory is released; each of
            // these waits is bounded too.
            for (long long j = issued > stages ? issued - stages : 0; j < issued; ++j)
                mbar_wait(&sm.full[j % stages], static_cast<unsigned>((j / stages) & 1));
        }
    } else {
        // ---------------- compute warps ----------------
        const int cw = warp - 1;
        const int r0 = cw * RPW;  // this warp's first row within a tile
        TileInputs cur{};
        if (n_my > 0) cur = load_tile_inputs<RPW>(p, tile_coord(p, cta), cw, lane);
        for (long long i = 0; i < n_my; ++i) {
            const int st = static_cast<int>(i % stages);
            const TileCoord c = tile_coord(p, cta + i * G);
            TileInputs nxt = cur;
            if (i + 1 < n_my)
                nxt = load_tile_inputs<RPW>(p, tile_coord(p, cta + (i + 1) * G), cw, lane);
            const bool ok = mbar_wait(&sm.full[st], static_cast<unsigned>((i / stages) & 1));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) atomicAdd(&p.err[2], 1u);
                break;
            }
            const long long s = sm.slot[st];
            // Read this warp's rows out of the stage, then hand the stage back.
            const float *stage = sm.buf + static_cast<size_t>(st) * p.rows_per_cta * kRowFloats;
            float4 v[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                v[r] = (s >= 0 && r0 + r < c.rows)
                           ? reinterpret_cast<const float4 *>(stage + (r0 + r) * kRowFloats)[lane]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            mbar_arrive(&sm.freed[st]);  // every lane: its reads precede the refill
            if (s >= 0) {
                const float dtv = softplus_f32(cur.dt + cur.bias);
                const float dA = expf(dtv * cur.A);
                float *srow = static_cast<float *>(p.state) + s * p.st_pool + c.h * p.st_head +
                              (c.row0 + r0) * p.st_row + lane * 4;
                float part[RPW];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const float xr = __shfl_sync(0xffffffffu, cur.x, r);
                    part[r] = update_cols(v[r], dA, dtv * xr, cur.bb, cur.cc);
                    if (r0 + r < c.rows)
                        __stcs(reinterpret_cast<float4 *>(srow + r * p.st_row), v[r]);
                }
                const float total = reduce_rows<RPW>(part, lane);
                const int rl = row_of_lane<RPW>(lane);
                const float xr = __shfl_sync(0xffffffffu, cur.x, rl);
                if (writes_row<RPW>(lane) && r0 + rl < c.rows)
                    p.out[c.b * p.out_b + c.h * p.out_h + c.row0 + r0 + rl] =
                        __float2bfloat16_rn(fmaf(cur.D, xr, total));
            }
            cur = nxt;
        }
    }
}

using BulkKernel = void (*)(SsuParams, BulkShape);

BulkKernel bulk_kernel(int rpw, bool idx64) {
    switch (rpw) {
        case 2: return idx64 ? ssu_bulk_kernel<2, true> : ssu_bulk_kernel<2, false>;
        case 4: return idx64 ? ssu_bulk_kernel<4, true> : ssu_bulk_kernel<4, false>;
        case 8: return idx64 ? ssu_bulk_kernel<8, true> : ssu_bulk_kernel<8, false>;
        case 16: return idx64 ? ssu_bulk_kernel<16, true> : ssu_bulk_kernel<16, false>;
        default: return nullptr;
    }
}

unsigned bulk_smem_bytes(int stages, int tile_rows) {
    return bulk_header_bytes(stages) + static_cast<unsigned>(stages) * tile_rows * kRowBytes;
}

}  // namespace
