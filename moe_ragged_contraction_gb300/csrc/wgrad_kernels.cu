// Ragged MXFP8 weight-gradient grouped GEMM for sm_103a.
//
// "Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on MI355X":
//   section 1  — dW[g] = dY[g]^T X[g]; offsets cut the contraction (token) axis;
//                A = dY^T [N,M], B = X^T [K,M] token-contiguous E4M3, one E8M0
//                scale per 32 tokens in planes [N,M/32] and [K,M/32];
//   section 4  — one CTA (here: one CTA pair) owns an output tile for its whole
//                reduction (no atomics, bit-reproducible);
//   section 5.3 — ragged runs: runtime length, 32-aligned start, empty experts
//                get an explicit zero store, scale reads stay in bounds;
//   section 5.4 — longest-expert-first order shortens the tail;
//   section 5.5 — bf16 narrowing (round to nearest even) in registers;
//   section 5.6 — scales re-laid out once per call before the main loop.
//
// Two kernels per call:
//   wgrad_prep : reads offs, clamps them, builds the schedule (per-expert
//                start / length / K-steps, longest-first order) and gathers
//                the scale bytes of every (128-row block of a tile, K-step)
//                into the 512-byte tcgen05 scale-factor block layout.
//   wgrad_main : persistent CTA pairs (2-CTA clusters, cta_group::2 MMAs),
//                warp-specialised: TMA producer, MMA issuer, stage watcher and
//                8 epilogue warps per CTA.
//
// Tiling. A pair tile is 256 rows of the "M-side" operand (split 128 / 128
// over the two CTAs and over TMEM lanes) by TN rows of the "N-side" operand
// (TN a multiple of 16, at most 448). Each 32-token chunk is one MMA of
// N1 = min(TN, 256) columns plus, for TN > 256, a second of N2 = TN - 256
// columns into the next TMEM columns; each CTA holds half of either MMA's
// N-side rows. The host picks which operand is the M side (A, rows n, by
// default; or B, rows k, the accumulator then holding the tile transposed)
// and TN from a cost model of the kernel (operand bytes per K-step against
// MMA cycles, padding, tile count).
//
// A K-step starts exactly at the group's first token (TMA coordinates need
// only 16-byte alignment, and 32 tokens are 32 bytes), so there is no leading
// partial step; the last step of a group issues only the ceil(rem/32) MMAs
// that cover its tokens, so bytes past the group end (the next expert's, or
// padding that may hold NaN) are loaded but never consumed.
#include <atomic>
#include <type_traits>

#include "mxw_internal.h"
#include "mxw_ptx.cuh"
#include "../../include/mxfp8_wgrad.h"

// 1: tiles wider than 256 columns (two MMAs per 32-token chunk, one A tile)
// read A from shared memory once per chunk through the collector buffer.
#ifndef MXW_COLLECTOR_A
#define MXW_COLLECTOR_A 1
#endif
// The producers of the persistent grid meet at the passes that follow a pass
// spanning two experts (pass_barrier_at): 1 always, 0 never, -1 where
// use_pass_barrier() predicts a gain.
#ifndef MXW_PASS_BARRIER
#define MXW_PASS_BARRIER -1
#endif
// Order of an expert's tiles: -1 the side with fewer rows fastest, 0 the N
// side's tiles fastest, 1 the M side's.
#ifndef MXW_ORDER
#define MXW_ORDER -1
#endif

namespace mxw {

__device__ int g_device_status = 0;

// ============================================================== prep kernel

constexpr int PREP_THREADS = 256;
constexpr int PREP_ROWS = 128;        // rows of one scale-factor block
constexpr int PREP_TILE_STEPS = 32;   // K-steps per gather task (one per lane)

// The block's contiguous share of the 16-byte-aligned interior of
// [p, p + bytes), streamed into L2 in 4 KB bulk prefetches (one per thread at
// a time). The gathers below read 128-byte pieces of rows that lie far apart;
// straight from DRAM such pieces each open a page and run at a fraction of
// the streaming rate, after this they hit L2. The few edge bytes outside the
// aligned interior are simply not prefetched (nothing outside the buffer is
// touched).
__device__ __forceinline__ void prefetch_share_l2(const uint8_t* p, size_t bytes) {
    constexpr size_t PIECE = 4096;
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15);
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(p) + bytes) & ~uintptr_t(15);
    if (bytes < 16 || a1 <= a0) return;
    const size_t n = a1 - a0;
    const size_t share = ((n + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
    const size_t lo = share * blockIdx.x;
    const size_t hi = lo + share < n ? lo + share : n;
    for (size_t o = lo + threadIdx.x * PIECE; o < hi; o += PREP_THREADS * PIECE)
        bulk_prefetch_l2(reinterpret_cast<const void*>(a0 + o), static_cast<uint32_t>(hi - o < PIECE ? hi - o : PIECE));
}

struct PrepSide {
    const uint8_t* plane;  // scale plane [rows][M/32]
    uint8_t* sf;           // scale-factor blocks [tiles][ts_max][blocks][512 B]
    int rows, tile_rows, tiles;
    int blocks;            // 128-row blocks per tile: ceil(tile_rows / 128)
};

// Four scale bytes starting at byte `off` of the plane (which holds `size`
// bytes), for rows at the end of a plane where an aligned word could run past
// it: four predicated byte loads (bytes at or past the end, or all four when
// `ok` is false, read as 0), no branch, so that a thread's loads for all its
// rows stay in flight together. Everywhere else the gathers read two aligned
// words and funnel-shift them (alignment taken on the absolute address, so an
// unaligned plane is fine: rounding down never leaves its allocation).
__device__ __forceinline__ uint32_t load_scale4_edge(const uint8_t* __restrict__ plane, size_t off, size_t size,
                                                     bool ok) {
    uint32_t v = 0;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        const bool in = ok && off + kb < size;
        const uint32_t b = in ? static_cast<uint32_t>(__ldg(plane + (in ? off + kb : 0))) : 0u;
        v |= b << (8 * kb);
    }
    return v;
}

// Every block first rebuilds the per-expert runs from offs (staged in shared
// memory by all threads, then scanned by one warp with shuffles; 3E + 1
// words of shared memory). Block 0 also writes the plan. Then the blocks
// stride over gather tasks (below), writing the 512-byte scale-factor blocks:
// block h of tile t of a side holds rows t * tile_rows + 128 h + r (r < 128;
// zero past the tile or the plane), and row r, 32-token block kb sits at byte
// (r % 32) * 16 + (r / 32) * 4 + kb. Blocks: the M side's tiles * blocks
// first, then the N side's.
__global__ void __launch_bounds__(PREP_THREADS) wgrad_prep(const int32_t* __restrict__ offs, const PrepSide sm_side,
                                                           const PrepSide sn_side, int32_t* __restrict__ plan, int E,
                                                           long long M, int ts_max, int grid, int prefetch) {
    extern __shared__ int prep_smem[];
    int* s_start = prep_smem;        // [E]
    int* s_end = s_start + E;        // [E]: raw offs first, then the clamped ends
    int* s_sb = s_end + E;           // [E + 1]: first global K-step of each expert, then the total
    __shared__ int s_flags;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    const int Mi = static_cast<int>(M);

    if (prefetch) {
        prefetch_share_l2(sm_side.plane, static_cast<size_t>(sm_side.rows) * static_cast<size_t>(M / 32));
        prefetch_share_l2(sn_side.plane, static_cast<size_t>(sn_side.rows) * static_cast<size_t>(M / 32));
    }
    // the main kernel may launch now: its prologue (barriers, TMEM, tensor
    // maps) overlaps this kernel, and it waits for this grid's completion (and
    // the visibility of its writes) before it reads the plan or the scales.
    // Every block of this grid is resident once all have passed here, so the
    // main kernel's CTAs only queue behind them for shared memory.
    griddep_launch_dependents();
    // On the global 128-token grid (grid != 0) the scale blocks do not depend
    // on the routing: only block 0 (the plan) reads offs, the others go
    // straight to the gather.
    const bool need_scan = !grid || blockIdx.x == 0;
    if (need_scan) {
        for (int g = threadIdx.x; g < E; g += PREP_THREADS) s_end[g] = offs[g];
        __syncthreads();
        if (warp == 0) {
            int carry_end = 0, carry_steps = 0, flags = 0;
            for (int base = 0; base < E; base += 32) {
                const int g = base + lane;
                int o = 0;
                if (g < E) {
                    o = s_end[g];
                    if (o < 0) { o = 0; flags |= MXFP8_DEV_OFFS_RANGE; }
                    if (o > Mi) { o = Mi; flags |= MXFP8_DEV_OFFS_RANGE; }
                    if (o & 31) { o &= ~31; flags |= MXFP8_DEV_OFFS_ALIGN; }
                }
                int m = o;  // inclusive running max -> clamped non-decreasing ends
    #pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    int t = __shfl_up_sync(full, m, d);
                    if (lane >= d) m = max(m, t);
                }
                const int end = max(m, carry_end);
                int start = __shfl_up_sync(full, end, 1);
                if (lane == 0) start = carry_end;
                if (g < E && o < start) flags |= MXFP8_DEV_OFFS_UNSORTED;
                const int ns = (end - start + BK - 1) / BK;
                int incl = ns;
    #pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    int t = __shfl_up_sync(full, incl, d);
                    if (lane >= d) incl += t;
                }
                __syncwarp();
                if (g < E) {
                    s_start[g] = start;
                    s_end[g] = end;
                    s_sb[g] = carry_steps + incl - ns;
                }
                carry_end = __shfl_sync(full, end, 31);
                carry_steps += __shfl_sync(full, incl, 31);
            }
    #pragma unroll
            for (int d = 16; d > 0; d >>= 1) flags |= __shfl_xor_sync(full, flags, d);
            if (lane == 0) {
                s_sb[E] = carry_steps;
                s_flags = flags;
            }
        }
        __syncthreads();
    }
    // K-steps the blocks cover: every expert's own steps, or the grid's
    const int TS = grid ? static_cast<int>((M + BK - 1) / BK) : s_sb[E];

    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            plan[0] = TS;
            plan[1] = E;
            plan[2] = 0;  // the main kernel's pass-barrier counter
            if (s_flags) atomicOr(&g_device_status, s_flags);
        }
        int32_t* ex = plan + PLAN_HDR;
        int32_t* order = ex + 4 * E;
        for (int g = threadIdx.x; g < E; g += PREP_THREADS) {
            const int len = s_end[g] - s_start[g];
            ex[4 * g + 0] = s_start[g];
            ex[4 * g + 1] = len;
            if (grid) {
                // K-steps on the global 128-token grid: the steps the run
                // touches, and the grid step of its first token
                ex[4 * g + 2] = len ? (s_start[g] + len + BK - 1) / BK - s_start[g] / BK : 0;
                ex[4 * g + 3] = s_start[g] / BK;
            } else {
                ex[4 * g + 2] = (len + BK - 1) / BK;
                ex[4 * g + 3] = s_sb[g];
            }
            int rank = 0;  // longest first; equal lengths keep expert order
            for (int h = 0; h < E; ++h) {
                const int lh = s_end[h] - s_start[h];
                rank += (lh > len) || (lh == len && h < g);
            }
            order[rank] = g;
        }
    }

    // Scale-factor gather as a tile transpose. A task is (128-row block, 32
    // consecutive global K-steps): lane l owns K-step gs0 + l, finds its
    // expert, and reads that step's (up to) 4 scale bytes of each row with one
    // or two aligned 32-bit loads, so a warp reads a contiguous run of each
    // row within an expert. The words are staged in a padded [128][33] shared
    // tile, then each 512-byte block is written by one warp with 16-byte
    // stores.
    uint32_t* tile = reinterpret_cast<uint32_t*>(s_sb + E + 1);  // [PREP_ROWS][PREP_TILE_STEPS + 1]
    const int nchunks = (TS + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS;
    const int mblocks = sm_side.tiles * sm_side.blocks;
    const int nblk = mblocks + sn_side.tiles * sn_side.blocks;
    const long long ntasks = static_cast<long long>(nblk) * nchunks;
    const long long sM = M / 32;
    // On the grid block 0 builds only the plan (its scan of offs would
    // otherwise delay its share of the gather: measured 4.1 against 3.3 us
    // for the other blocks at the 16B shape); the other blocks gather.
    const bool plan_only = grid && gridDim.x > 1;
    const long long tstride = plan_only ? gridDim.x - 1 : gridDim.x;
    for (long long task = plan_only ? static_cast<long long>(blockIdx.x) - 1 : blockIdx.x; task < ntasks;
         task += tstride) {
        if (task < 0) break;
        const int hb = static_cast<int>(task / nchunks);
        const int gs0 = static_cast<int>(task - static_cast<long long>(hb) * nchunks) * PREP_TILE_STEPS;
        const bool mside = hb < mblocks;
        const uint8_t* plane = mside ? sm_side.plane : sn_side.plane;
        uint8_t* sf = mside ? sm_side.sf : sn_side.sf;
        const int rows = mside ? sm_side.rows : sn_side.rows;
        const int tile_rows = mside ? sm_side.tile_rows : sn_side.tile_rows;
        const int blocks = mside ? sm_side.blocks : sn_side.blocks;
        const int local = mside ? hb : hb - mblocks;
        const int t = local / blocks, h = local - t * blocks;
        const int in_tile0 = PREP_ROWS * h;  // first row of this block inside its tile
        const int row0 = t * tile_rows + in_tile0;
        // this lane's K-step: its expert, first scale column and valid 32-token blocks
        const int gs = gs0 + lane;
        long long col = 0;
        int nvalid = 0;
        if (gs < TS && grid) {
            // grid step gs: 32-token blocks 4 gs .. 4 gs + 3 of every row
            col = 4LL * gs;
            const long long left = M / 32 - col;
            nvalid = static_cast<int>(left < 4 ? left : 4);
        } else if (gs < TS) {
            int lo = 0, hi = E;  // expert owning gs: the last g with s_sb[g] <= gs
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_sb[mid] <= gs) lo = mid; else hi = mid;
            }
            const long long t0 = static_cast<long long>(s_start[lo]) + static_cast<long long>(gs - s_sb[lo]) * BK;
            col = t0 >> 5;
            const long long left = (static_cast<long long>(s_end[lo]) - t0 + 31) >> 5;
            nvalid = static_cast<int>(left < 4 ? left : 4);
        }
        const uint32_t keep = nvalid >= 4 ? 0xffffffffu : ((1u << (8 * nvalid)) - 1u);
        const size_t plane_bytes = static_cast<size_t>(rows) * static_cast<size_t>(sM);
        constexpr int ROWS_PER_WARP = PREP_ROWS / (PREP_THREADS / 32);
        // rows of the plane this block may read: inside its tile and the plane
        const int rows_lim = min(rows, row0 - in_tile0 + tile_rows);
        uint32_t wv[ROWS_PER_WARP];
        // on the grid with 4-byte-aligned rows every step's 4 scale bytes are
        // one aligned word: one load per row
        const bool words = grid && ((reinterpret_cast<uintptr_t>(plane) | static_cast<uintptr_t>(sM)) & 3) == 0;
        if (words && nvalid > 0 && static_cast<size_t>(rows_lim - 1) * sM + col + 4 <= plane_bytes) {
            uint32_t v[ROWS_PER_WARP];
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int row = min(row0 + warp + i * (PREP_THREADS / 32), rows_lim - 1);
                v[i] = __ldg(reinterpret_cast<const uint32_t*>(plane + static_cast<size_t>(row) * sM + col));
            }
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int row = row0 + warp + i * (PREP_THREADS / 32);
                wv[i] = row < rows_lim ? (v[i] & keep) : 0u;
            }
        } else if (nvalid > 0 && static_cast<size_t>(rows_lim - 1) * sM + col + 8 <= plane_bytes) {
            // every word this lane reads lies inside the plane: rows past the
            // limit read the last valid row and are zeroed afterwards
            // all loads first, then the shifts: the words of every row in flight together
            uint32_t lo[ROWS_PER_WARP], hi[ROWS_PER_WARP], sh[ROWS_PER_WARP];
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int row = min(row0 + warp + i * (PREP_THREADS / 32), rows_lim - 1);
                const uintptr_t a = reinterpret_cast<uintptr_t>(plane) + static_cast<size_t>(row) * sM + col;
                const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
                lo[i] = __ldg(w);
                hi[i] = __ldg(w + 1);
                sh[i] = static_cast<uint32_t>(a & 3) * 8;
            }
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int row = row0 + warp + i * (PREP_THREADS / 32);
                wv[i] = row < rows_lim ? (__funnelshift_r(lo[i], hi[i], sh[i]) & keep) : 0u;
            }
        } else {
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int row = row0 + warp + i * (PREP_THREADS / 32);
                const bool ok = nvalid > 0 && row < rows_lim;
                wv[i] = load_scale4_edge(plane, ok ? static_cast<size_t>(row) * sM + col : 0, plane_bytes, ok) & keep;
            }
        }
#pragma unroll
        for (int i = 0; i < ROWS_PER_WARP; ++i)
            tile[(warp + i * (PREP_THREADS / 32)) * (PREP_TILE_STEPS + 1) + lane] = wv[i];
        __syncthreads();
        // block j of this task: lane r0 writes rows r0, r0+32, r0+64, r0+96 (16 bytes)
        for (int j = warp; j < PREP_TILE_STEPS; j += PREP_THREADS / 32) {
            if (gs0 + j >= TS) continue;
            uint4 o;
            o.x = tile[(lane + 0) * (PREP_TILE_STEPS + 1) + j];
            o.y = tile[(lane + 32) * (PREP_TILE_STEPS + 1) + j];
            o.z = tile[(lane + 64) * (PREP_TILE_STEPS + 1) + j];
            o.w = tile[(lane + 96) * (PREP_TILE_STEPS + 1) + j];
            uint8_t* dst = sf + ((static_cast<size_t>(t) * ts_max + gs0 + j) * blocks + h) * SF_ATOM;
            reinterpret_cast<uint4*>(dst)[lane] = o;
        }
        __syncthreads();
    }
}

// ============================================================== grouped GEMM prep

// Plan and scale re-layout of the grouped GEMM (the non-contracting ragged
// dot: "Group-GEMM in XLA", Part 1; the forward and data-gradient products of
// the expert layer): rows [offs[g-1], offs[g]) of X multiply W[g]. Every
// block rebuilds the per-expert row runs from offs (clamped into [0, M],
// non-decreasing) and their 256-row tiles; block 0 writes the plan: [0] items
// (row tiles x N-side tiles), [1] E, [2] row tiles, then one int4 per row
// tile (expert, first row, end of the expert's rows, 0). Then the blocks
// gather scale-factor blocks for (row tile, half) and (expert, N-side tile,
// 128-row block), one K-step each, and zero the output rows past the last
// group.
struct GemmPrepArgs {
    const int32_t* offs;
    const uint8_t *sX, *sW;    // [M][K/32], [E][N][K/32]
    uint8_t *sfm, *sfn;        // [row tiles][ksteps][2][512], [E * tiles_n][ksteps][nblk][512]
    int32_t* plan;
    uint16_t* out;             // [M][N]
    int E, N, K, ksteps, tn, tiles_n, nblk, mtiles_max;
    long long M;
};

__global__ void __launch_bounds__(PREP_THREADS) gemm_prep(const GemmPrepArgs a) {
    extern __shared__ int prep_smem[];
    int* s_start = prep_smem;        // [E]
    int* s_end = s_start + a.E;      // [E]
    int* s_mtb = s_end + a.E;        // [E + 1]: first row tile of each expert, then the total
    __shared__ int s_flags;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    const int E = a.E;
    const long long M = a.M;

    prefetch_share_l2(a.sX, static_cast<size_t>(M) * static_cast<size_t>(a.K / 32));
    prefetch_share_l2(a.sW, static_cast<size_t>(E) * a.N * static_cast<size_t>(a.K / 32));
    griddep_launch_dependents();  // as in wgrad_prep: the main kernel's prologue overlaps this grid
    for (int g = threadIdx.x; g < E; g += PREP_THREADS) s_end[g] = a.offs[g];
    __syncthreads();
    if (warp == 0) {
        long long carry_end = 0;
        int carry_tiles = 0, flags = 0;
        for (int base = 0; base < E; base += 32) {
            const int g = base + lane;
            long long o = 0;
            if (g < E) {
                o = s_end[g];
                if (o < 0) { o = 0; flags |= MXFP8_DEV_OFFS_RANGE; }
                if (o > M) { o = M; flags |= MXFP8_DEV_OFFS_RANGE; }
            }
            long long m = o;  // inclusive running max -> clamped non-decreasing ends
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const long long t = __shfl_up_sync(full, m, d);
                if (lane >= d) m = max(m, t);
            }
            const long long end = max(m, carry_end);
            long long start = __shfl_up_sync(full, end, 1);
            if (lane == 0) start = carry_end;
            if (g < E && o < start) flags |= MXFP8_DEV_OFFS_UNSORTED;
            const int nt = static_cast<int>((end - start + 2 * BM - 1) / (2 * BM));
            int incl = nt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int t = __shfl_up_sync(full, incl, d);
                if (lane >= d) incl += t;
            }
            __syncwarp();
            if (g < E) {
                s_start[g] = static_cast<int>(start);
                s_end[g] = static_cast<int>(end);
                s_mtb[g] = carry_tiles + incl - nt;
            }
            carry_end = __shfl_sync(full, end, 31);
            carry_tiles += __shfl_sync(full, incl, 31);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) flags |= __shfl_xor_sync(full, flags, d);
        if (lane == 0) {
            s_mtb[E] = carry_tiles;
            s_flags = flags;
        }
    }
    __syncthreads();
    const int mtiles = s_mtb[E];

    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            a.plan[0] = mtiles * a.tiles_n;
            a.plan[1] = E;
            a.plan[2] = mtiles;
            if (s_flags) atomicOr(&g_device_status, s_flags);
        }
        int4* ent = reinterpret_cast<int4*>(a.plan + PLAN_HDR);
        for (int g = threadIdx.x; g < E; g += PREP_THREADS)
            for (int j = 0, mt = s_mtb[g]; mt < s_mtb[g + 1]; ++j, ++mt)
                ent[mt] = make_int4(g, s_start[g] + 2 * BM * j, s_end[g], 0);
    }

    // scale-factor gather: tasks (128-row block, 32 consecutive K-steps), the
    // row tiles' halves first, then the (expert, N-side tile) blocks
    uint32_t* tile = reinterpret_cast<uint32_t*>(s_mtb + E + 1);  // [PREP_ROWS][PREP_TILE_STEPS + 1]
    const int nchunks = (a.ksteps + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS;
    const int mblocks = 2 * mtiles;
    const long long nblk_total = static_cast<long long>(mblocks) + static_cast<long long>(E) * a.tiles_n * a.nblk;
    const long long ntasks = nblk_total * nchunks;
    const long long sK = a.K / 32;
    for (long long task = blockIdx.x; task < ntasks; task += gridDim.x) {
        const long long hb = task / nchunks;
        const int s0 = static_cast<int>(task - hb * nchunks) * PREP_TILE_STEPS;
        const bool mside = hb < mblocks;
        const uint8_t* plane;
        uint8_t* dst0;  // block of K-step 0; consecutive K-steps `stride` bytes apart
        size_t stride, plane_bytes;
        long long row0;
        int rows_valid;  // rows of this 128-row block that exist
        if (mside) {
            const int mt = static_cast<int>(hb >> 1), h = static_cast<int>(hb & 1);
            int lo = 0, hi = E;  // expert of row tile mt: the last g with s_mtb[g] <= mt
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_mtb[mid] <= mt) lo = mid; else hi = mid;
            }
            row0 = static_cast<long long>(s_start[lo]) + 2LL * BM * (mt - s_mtb[lo]) + PREP_ROWS * h;
            const long long left = s_end[lo] - row0;
            rows_valid = static_cast<int>(left < 0 ? 0 : (left > PREP_ROWS ? PREP_ROWS : left));
            plane = a.sX;
            plane_bytes = static_cast<size_t>(M) * sK;
            dst0 = a.sfm + (static_cast<size_t>(mt) * a.ksteps * 2 + h) * SF_ATOM;
            stride = 2 * SF_ATOM;
        } else {
            const long long nb = hb - mblocks;  // (g * tiles_n + tn) * nblk + h
            const int h = static_cast<int>(nb % a.nblk);
            const long long gt = nb / a.nblk;
            const int g = static_cast<int>(gt / a.tiles_n), tn = static_cast<int>(gt % a.tiles_n);
            const int in_tile0 = PREP_ROWS * h;
            row0 = static_cast<long long>(tn) * a.tn + in_tile0;
            const long long left = min(static_cast<long long>(a.tn - in_tile0), static_cast<long long>(a.N) - row0);
            rows_valid = static_cast<int>(left < 0 ? 0 : (left > PREP_ROWS ? PREP_ROWS : left));
            plane = a.sW + static_cast<size_t>(g) * a.N * sK;
            plane_bytes = static_cast<size_t>(a.N) * sK;
            dst0 = a.sfn + (static_cast<size_t>(gt) * a.ksteps * a.nblk + h) * SF_ATOM;
            stride = static_cast<size_t>(a.nblk) * SF_ATOM;
        }
        const int s = s0 + lane;  // this lane's K-step
        int nvalid = 0;
        if (s < a.ksteps) {
            const int left = (a.K - s * BK + 31) >> 5;
            nvalid = left < 4 ? left : 4;
        }
        const uint32_t keep = nvalid >= 4 ? 0xffffffffu : ((1u << (8 * nvalid)) - 1u);
        constexpr int ROWS_PER_WARP = PREP_ROWS / (PREP_THREADS / 32);
        uint32_t wv[ROWS_PER_WARP];
        if (nvalid > 0 && rows_valid > 0 &&
            static_cast<size_t>(row0 + rows_valid - 1) * sK + 4 * s + 8 <= plane_bytes) {
            // all of this lane's words inside the plane (see wgrad_prep)
            uint32_t lo[ROWS_PER_WARP], hi[ROWS_PER_WARP], sh[ROWS_PER_WARP];
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int r = min(warp + i * (PREP_THREADS / 32), rows_valid - 1);
                const uintptr_t ad = reinterpret_cast<uintptr_t>(plane) + static_cast<size_t>(row0 + r) * sK + 4 * s;
                const uint32_t* w = reinterpret_cast<const uint32_t*>(ad & ~uintptr_t(3));
                lo[i] = __ldg(w);
                hi[i] = __ldg(w + 1);
                sh[i] = static_cast<uint32_t>(ad & 3) * 8;
            }
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int r = warp + i * (PREP_THREADS / 32);
                wv[i] = r < rows_valid ? (__funnelshift_r(lo[i], hi[i], sh[i]) & keep) : 0u;
            }
        } else {
#pragma unroll
            for (int i = 0; i < ROWS_PER_WARP; ++i) {
                const int r = warp + i * (PREP_THREADS / 32);
                const bool ok = nvalid > 0 && r < rows_valid;
                wv[i] = load_scale4_edge(plane, ok ? static_cast<size_t>(row0 + r) * sK + 4 * s : 0, plane_bytes, ok) & keep;
            }
        }
#pragma unroll
        for (int i = 0; i < ROWS_PER_WARP; ++i)
            tile[(warp + i * (PREP_THREADS / 32)) * (PREP_TILE_STEPS + 1) + lane] = wv[i];
        __syncthreads();
        for (int j = warp; j < PREP_TILE_STEPS; j += PREP_THREADS / 32) {
            if (s0 + j >= a.ksteps) continue;
            uint4 o;
            o.x = tile[(lane + 0) * (PREP_TILE_STEPS + 1) + j];
            o.y = tile[(lane + 32) * (PREP_TILE_STEPS + 1) + j];
            o.z = tile[(lane + 64) * (PREP_TILE_STEPS + 1) + j];
            o.w = tile[(lane + 96) * (PREP_TILE_STEPS + 1) + j];
            reinterpret_cast<uint4*>(dst0 + static_cast<size_t>(s0 + j) * stride)[lane] = o;
        }
        __syncthreads();
    }
    // rows past the last group belong to no expert: exact zeros
    {
        const long long end_last = E > 0 ? s_end[E - 1] : 0;
        const long long n_zero = (M - end_last) * a.N;  // N % 8 == 0: 16-byte runs
        uint4* z = reinterpret_cast<uint4*>(a.out + end_last * a.N);
        for (long long i = static_cast<long long>(blockIdx.x) * PREP_THREADS + threadIdx.x; i < n_zero / 8;
             i += static_cast<long long>(gridDim.x) * PREP_THREADS)
            z[i] = make_uint4(0, 0, 0, 0);
    }
}

// ============================================================== main kernel

// One CTA pair (a 2-CTA cluster) owns a 256 x TN output tile. CTA r of the
// pair holds M-side rows tm*256 + 128r .. +128 and half of the N-side rows of
// each MMA (rows r*N1/2 .. +N1/2 and N1 + r*N2/2 .. +N2/2 of the tile) in its
// shared memory, its own 128 accumulator rows in its TMEM, and stores those
// 128 rows of the tile. The leader (r = 0) issues the M = 256 block-scaled
// MMAs for both; each SM then reads 16 KB + TN * 64 bytes of operands per
// K-step for 128 x TN x 128 multiply-adds.
//
// Shared memory (runtime-sized rings of `stages` entries, each 1024-byte
// aligned where the 128-byte swizzle needs it): M-side tiles [stages][16 KB],
// N-side tiles [stages][TN/2 * 128 B], M-side scale blocks [stages][512 B],
// N-side scale blocks [stages][nblk_n * 512 B], then the mbarriers.
// TMEM (512 columns): accumulator columns [0, TN); from column TN on,
// `sf_slots` scale-factor slots of 4 + 4 * nblk_n columns (M-side block,
// then the N-side blocks).
constexpr int PAIR_M = 2 * BM;        // 256 M-side rows per pair tile
constexpr int A_STAGE = BM * BK;      // M-side operand: this CTA's 128 rows (16 KB)
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 3;                        // producer, MMA issuer, stage watcher, then the epilogue
constexpr int MAIN_THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int MAX_STAGES = 7;
constexpr uint32_t STG_CHUNK = 32 * 64;  // one epilogue chunk: 32 rows x 32 bf16 columns (64-byte swizzle)
constexpr int MAIN_SMEM_MAX = 232448;  // the sm_100-family opt-in limit per CTA
// Named barriers between the stage watcher and the MMA warp (64 threads each):
// BAR_READY + st: stage st holds data (watcher arrives, MMA warp syncs);
// BAR_FREE + st: the MMA warp has taken stage st (MMA warp arrives, watcher
// syncs before it signals that stage again), so arrivals and syncs on every
// id pair up one to one.
constexpr uint32_t BAR_READY = 1;
constexpr uint32_t BAR_FREE = 8;
constexpr uint32_t TMEM_COLS = 512;

static_assert(BAR_READY + MAX_STAGES <= BAR_FREE && BAR_FREE + MAX_STAGES <= 16, "named barrier ids");
static_assert(MAX_TN <= 448 && MAX_TN % 16 == 0, "N-side tile: at most two MMAs (256 + 192 columns)");

// Instruction descriptor, kind::mxf8f6f4: A and B E4M3 (0), both K-major,
// E8M0 scales (bit 23), M >> 4 at bits 24-28 (M = 256 across the pair). N >> 3
// (bits 17-22) is or-ed in per MMA width, the scale byte selectors for B
// (bits 4-5) and A (bits 29-30) per 32-token chunk.
constexpr uint32_t IDESC_BASE = (1u << 23) | (static_cast<uint32_t>(PAIR_M >> 4) << 24);

struct MainParams {
    const int32_t* plan;
    uint16_t* out;
    int mode;                // 0: weight gradient (contraction over ragged token runs); 1: grouped GEMM (ragged rows)
    int E, N, K;             // mode 0: out[E][N][K]; mode 1: out[M][N], K the contracted length
    long long out_stride;    // elements between output rows (rows of the 256-row side)
    int col_limit;           // valid output columns (columns of the tn side)
    int ksteps;              // mode 1: K-steps of every tile
    int ts_max;
    int tiles_m, tiles_n;    // pair tiles along the M side (256 rows) and the N side (tn rows)
    int tn, n1, n2;          // N-side tile rows = n1 + n2 (the two MMA widths; n2 may be 0)
    int nblk_n;              // 128-row scale blocks per N-side tile
    int kn;                  // 0: M side = rows of A (n), N side = rows of B (k); 1: swapped
    int m_fastest;           // mode 0: an expert's tiles ordered M-side tile fastest (else N-side tile fastest)
    int grid;                // mode 0: K-steps on the global 128-token grid (scale blocks per grid step)
    int pass_bar;            // mode 0: producers meet at the passes that follow one spanning two experts
    unsigned int* pass_ctr;  // their arrival counter (zeroed by the prep kernel)
    int stages, sf_slots;
    int acc_bufs;            // accumulators in TMEM (2: the next tile's MMAs overlap this tile's drain)
    int wide_stores;         // 32-byte output stores (rows of 16 columns 32-byte aligned), else 16-byte
    int tma_store;           // epilogue chunks through shared memory and TMA stores (transposed tiles: weight gradient only)
    int stg_bufs;            // staging buffers per epilogue warp (1 or 2) when tma_store
    uint32_t sf_col0;        // first TMEM column of the scale-factor slots
    uint32_t off_b, off_sfa, off_sfb, off_stg, off_bar, b_stage;  // shared-memory layout (bytes)
    unsigned long long wait_ns;
    int stall_first_stage;   // test hook: over-declare the first stage's bytes so its wait runs out
};

__device__ uint32_t g_suspend_ns = 0;  // try_wait suspend hint for waiting roles (0: plain polling)

// Bounded wait: returns false (and raises the CTA's abort flag and the device
// status word) if the phase does not complete within wait_ns, or returns
// false at once if another role of this CTA already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned long long wait_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    const uint32_t hint = g_suspend_ns;
    for (;;) {
        if (hint ? mbar_try_wait_suspend(bar, parity, hint) : mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > wait_ns) {
            *abort_flag = 1;
            atomicOr(&g_device_status, MXFP8_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait used while tearing down (ignores the abort flag).
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, unsigned long long wait_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > wait_ns) {
            atomicOr(&g_device_status, MXFP8_DEV_WAIT_TIMEOUT);
            return;
        }
    }
}

struct Item {
    int g, tm, tn;        // expert, M-side and N-side tile
    int start, len;       // contraction: first coordinate and length
    int nsteps;           // K-steps
    int kk0;              // 32-token chunks of the first K-step before the run's first token (grid K-steps)
    int m0, m_end;        // M-side rows of the tile start at m0; rows at or past m_end are not stored
    int sfm, sfn;         // scale-factor block rows of the tile's first K-step (M side: this CTA adds its rank)
    int z;                // N-side tensor-map depth coordinate (the expert in the grouped GEMM)
    long long orow0;      // output row of M-side row 0 (rows of the 256 side)
};

// Work item i -> expert and pair tile.
// Mode 0 (weight gradient): items in longest-expert-first order, the tiles of
// one expert consecutive, N-side tiles fastest; plan entries per expert.
// Mode 1 (grouped GEMM): item = (row tile, N-side tile), N-side fastest; the
// plan holds one entry per row tile: (expert, first row, end of the expert's rows).
__device__ __forceinline__ Item load_item(const MainParams& p, long long i) {
    Item it;
    if (p.mode == 0) {
        const int32_t* ex = p.plan + PLAN_HDR;
        const int32_t* order = ex + 4 * p.E;
        const int ntpe = p.tiles_m * p.tiles_n;
        const int r = static_cast<int>(i / ntpe);
        const int t = static_cast<int>(i - static_cast<long long>(r) * ntpe);
        it.g = __ldg(order + r);
        if (p.m_fastest) {
            it.tn = t / p.tiles_m;
            it.tm = t - it.tn * p.tiles_m;
        } else {
            it.tm = t / p.tiles_n;
            it.tn = t - it.tm * p.tiles_n;
        }
        const int start = __ldg(ex + 4 * it.g + 0);
        const int len = __ldg(ex + 4 * it.g + 1);
        // grid K-steps start at the run's 128-token grid step; its leading
        // chunks belong to the run before and are skipped
        const int lead = p.grid ? (start & (BK - 1)) : 0;
        it.start = start - lead;
        it.len = len + lead;
        it.kk0 = lead >> 5;
        it.nsteps = __ldg(ex + 4 * it.g + 2);
        const int sb = __ldg(ex + 4 * it.g + 3);
        it.m0 = it.tm * (2 * BM);
        it.m_end = p.kn ? p.K : p.N;
        it.sfm = (it.tm * p.ts_max + sb) * 2;
        it.sfn = (it.tn * p.ts_max + sb) * p.nblk_n;
        it.z = 0;
        it.orow0 = static_cast<long long>(it.g) * p.N;
    } else {
        const int mt = static_cast<int>(i / p.tiles_n);
        it.tn = static_cast<int>(i - static_cast<long long>(mt) * p.tiles_n);
        const int4 e = __ldg(reinterpret_cast<const int4*>(p.plan + PLAN_HDR) + mt);
        it.g = e.x;
        it.tm = mt;
        it.m0 = e.y;
        it.m_end = e.z;
        it.start = 0;
        it.len = p.K;
        it.kk0 = 0;
        it.nsteps = p.ksteps;
        it.sfm = mt * p.ksteps * 2;
        it.sfn = (it.g * p.tiles_n + it.tn) * p.ksteps * p.nblk_n;
        it.z = it.g;
        it.orow0 = 0;
    }
    return it;
}

// Static schedule over CTA pairs: pass p hands items [p*G, (p+1)*G) to the
// pairs, reversing the direction on odd passes so that, with items sorted by
// cost, the loads even out (no atomics; a pair knows its items from its
// index alone, and both CTAs of a pair walk the same list).
__device__ __forceinline__ long long item_index(long long pass, int G, int pair) {
    return pass * G + ((pass & 1) ? (G - 1 - pair) : pair);
}

// Next item of this pair's static schedule at or after pass `pass` (which is
// advanced past it), or -1 when the schedule is exhausted.
__device__ __forceinline__ long long next_item(long long& pass, int G, int pair, long long total) {
    while (pass * G < total) {
        const long long i = item_index(pass, G, pair);
        ++pass;
        if (i < total) return i;
    }
    return -1;
}

// Whether the producers meet before pass q of the static schedule (q >= 1):
// pass q is full (every pair has an item in it) and pass q - 1 spans an
// expert boundary (items of two experts, possibly of different lengths).
__device__ __forceinline__ bool pass_barrier_at(long long q, int G, long long total, int ntpe) {
    if (q < 1 || (q + 1) * G > total) return false;
    return ((q - 1) * G) / ntpe != (q * G - 1) / ntpe;
}

// Grid barrier among the producers (one lane per CTA): arrive, then wait
// until `target` arrivals; bounded like every other wait here.
__device__ __forceinline__ bool pass_barrier_wait(unsigned int* ctr, unsigned int target, volatile int* abort_flag,
                                                  unsigned long long wait_ns) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > wait_ns) {
            *abort_flag = 1;
            atomicOr(&g_device_status, MXFP8_DEV_WAIT_TIMEOUT);
            return false;
        }
        __nanosleep(128);
    }
}

// This pair's items in schedule order, the next item's plan entry loaded one
// item ahead so that its global-memory latency overlaps the current item.
struct ItemStream {
    const MainParams& p;
    int G, pair;
    long long total, pass, i_next, cur;  // cur: index of the item next() returned last
    Item it_next;

    __device__ __forceinline__ ItemStream(const MainParams& p_, int G_, int pair_, long long total_)
        : p(p_), G(G_), pair(pair_), total(total_), pass(0), cur(-1) {
        i_next = next_item(pass, G, pair, total);
        if (i_next >= 0) it_next = load_item(p, i_next);
    }

    __device__ __forceinline__ bool next(Item& it) {
        if (i_next < 0) return false;
        it = it_next;
        cur = i_next;
        i_next = next_item(pass, G, pair, total);
        if (i_next >= 0) it_next = load_item(p, i_next);
        return true;
    }
};

// State the MMA issuer needs besides the kernel parameters.
struct MmaCtx {
    uint32_t tmem, sbase, bar_empty, bar_tfull, bar_tempty, bar_drain;  // tfull / tempty: one per accumulator
    volatile int* abort_flag;
    int lane, G, pair;
    long long total;
    int nt_per_expert;
};

// MMA issuer of the leader CTA, for N-side tiles of NBLK 128-row scale blocks
// (NBLK > 2: two MMAs per 32-token chunk, the first 256 wide). The whole warp
// walks the schedule; one elected lane issues each tcgen05 operation. The
// per-stage loop reads no memory and takes no data-dependent branch between
// tcgen05 operations (the block count is a template parameter, everything
// else sits in registers): a load, a constant-bank read of a kernel parameter
// or an mbarrier probe here stalls the warp long enough to drain the tensor
// pipe, so stage readiness arrives through named barriers from the watcher
// warp. After an abort the loop still walks every stage (skipping the tensor
// work) so that the named barriers stay paired.
template <int NBLK>
__device__ __forceinline__ void mma_issue(const MainParams& p, const MmaCtx& x) {
    constexpr bool TWO = NBLK > 2;
    constexpr uint32_t SF_COLS = 4u + 4u * NBLK;
    constexpr uint32_t SFB_STAGE = NBLK * SF_ATOM;
    constexpr uint32_t B2_OFF = 128u * BK;  // second MMA's rows follow the first's 128 per CTA
    const int lane = x.lane;
    const uint32_t tmem = x.tmem;
    const uint32_t idesc1 = in_reg(IDESC_BASE | (static_cast<uint32_t>(p.n1 >> 3) << 17));
    const uint32_t idesc2 = in_reg(IDESC_BASE | (static_cast<uint32_t>(p.n2 >> 3) << 17));
    const uint32_t nstages = in_reg(static_cast<uint32_t>(p.stages));
    const uint32_t nslots = in_reg(static_cast<uint32_t>(p.sf_slots));
    const uint32_t sf_tmem0 = in_reg(tmem + p.sf_col0);
    const uint32_t nbuf = in_reg(static_cast<uint32_t>(p.acc_bufs));
    const uint32_t acc_cols = in_reg(static_cast<uint32_t>(p.tn));
    const uint32_t a_s0 = in_reg(x.sbase);
    const uint32_t sfa_s0 = in_reg(x.sbase + p.off_sfa);
    const uint32_t sfb_s0 = in_reg(x.sbase + p.off_sfb);
    const uint32_t b_s0 = in_reg(x.sbase + p.off_b);
    const uint32_t b_stage = in_reg(p.b_stage);
    uint32_t c = 0;
    uint32_t st = 0, slot = 0, buf = 0, acc_phase = 0;  // accumulator buffer of the current tile and its use count parity
    bool live = true;
    ItemStream items(p, x.G, x.pair, x.total);
    Item it;
    while (items.next(it)) {
        if (it.nsteps == 0) continue;
        if (live) {
            bool ok = true;
            // both CTAs' epilogues have drained the accumulator; their arrivals
            // only signal (the drained TMEM loads completed before them), so a
            // CTA-scope acquire is enough
            if (lane == 0)
                ok = !*x.abort_flag && wait_phase(x.bar_tempty + 8 * buf, acc_phase ^ 1, x.abort_flag, p.wait_ns);
            live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        tc_fence_after();
        const uint32_t acc_t = tmem + buf * acc_cols;
        // scale factors of stage `stg` into TMEM slot `slt`
        auto copy_sf = [&](uint32_t stg, uint32_t slt) {
            const uint32_t sfa_t = sf_tmem0 + slt * SF_COLS;
            tc_cp_32x128b_warpx4_pair_elect(sfa_t, desc_sf_block(sfa_s0 + stg * SF_ATOM));
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
                tc_cp_32x128b_warpx4_pair_elect(sfa_t + 4 + 4 * b, desc_sf_block(sfb_s0 + stg * SFB_STAGE + b * SF_ATOM));
        };
        // the MMAs of 32-token chunk kk of K-step s from stage stg, scales in slot slt
        auto mma_chunk = [&](int s, int kk, uint32_t stg, uint32_t slt) {
            const uint32_t sfa_t = sf_tmem0 + slt * SF_COLS;
            const uint32_t sfb_t = sfa_t + 4;
            const uint32_t a_s = a_s0 + stg * A_STAGE;
            const uint32_t b_s = b_s0 + stg * b_stage;
            const uint32_t sel = (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
            const uint32_t acc = (s > 0 || kk > it.kk0) ? 1u : 0u;
            const uint64_t ad = desc_kmajor_sw128(a_s + 32 * kk);
            if (TWO && MXW_COLLECTOR_A) {
                // both MMAs of the chunk multiply the same A tile: the
                // second reads it from the collector buffer
                tc_mma_mxf8_pair_elect_fill(acc_t, ad, desc_kmajor_sw128(b_s + 32 * kk), idesc1 | sel, sfa_t, sfb_t,
                                            acc);
                tc_mma_mxf8_pair_elect_lastuse(acc_t + 256, ad, desc_kmajor_sw128(b_s + B2_OFF + 32 * kk),
                                               idesc2 | sel, sfa_t, sfb_t + 8, acc);
            } else {
                tc_mma_mxf8_pair_elect(acc_t, ad, desc_kmajor_sw128(b_s + 32 * kk), idesc1 | sel, sfa_t, sfb_t, acc);
                if (TWO)
                    tc_mma_mxf8_pair_elect(acc_t + 256, ad, desc_kmajor_sw128(b_s + B2_OFF + 32 * kk), idesc2 | sel,
                                           sfa_t, sfb_t + 8, acc);
            }
        };
        for (int s = 0; s < it.nsteps; ++s, ++c) {
            named_bar_sync(BAR_READY + st, 64);
            if (live) {
                tc_fence_after();
                copy_sf(st, slot);
                const int rem = it.len - s * BK;
                const int nk = rem >= BK ? 4 : (rem >> 5);
                for (int kk = s == 0 ? it.kk0 : 0; kk < nk; ++kk) mma_chunk(s, kk, st, slot);
                tc_commit_pair_elect(x.bar_empty + 8 * st, 0x3);  // frees the stage in both CTAs
            }
            named_bar_arrive(BAR_FREE + st, 64);
            if (++st == nstages) st = 0;
            if (++slot == nslots) slot = 0;
        }
        if (live) {
            tc_commit_pair_elect(x.bar_tfull + 8 * buf, 0x3);  // both accumulator halves complete
            if (++buf == nbuf) {
                buf = 0;
                acc_phase ^= 1;
            }
        }
    }
    // every MMA / copy issued for the pair has finished before teardown
    tc_commit_pair_elect(x.bar_drain, 0x3);
}

// maps: M-side operand (boxes of 128 rows x BK tokens), N-side operand for the
// first MMA (n1/2 rows) and for the second (n2/2 rows; unused when n2 == 0),
// the two sides' scale-factor blocks as u32 [blocks][128] (boxes of 1 and
// nblk_n blocks), and the bf16 output as [depth][rows][columns] (boxes of 32 x
// 32 x 1, 64-byte swizzle; used only when p.tma_store).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MAIN_THREADS, 1)
    wgrad_main(const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmN1,
               const __grid_constant__ CUtensorMap tmN2, const __grid_constant__ CUtensorMap tmSFM,
               const __grid_constant__ CUtensorMap tmSFN, const __grid_constant__ CUtensorMap tmOut,
               const MainParams p) {
    extern __shared__ uint8_t main_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(main_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs), 1 = peer
    const bool leader = rank == 0;
    const int S = p.stages;
    const uint32_t sfb_stage = static_cast<uint32_t>(p.nblk_n) * SF_ATOM;

    const uint32_t bar_full = sbase + p.off_bar;
    const uint32_t bar_empty = bar_full + 8 * S;
    const uint32_t bar_tfull = bar_empty + 8 * S;   // [2]
    const uint32_t bar_tempty = bar_tfull + 16;     // [2]
    const uint32_t bar_drain = bar_tempty + 16;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_bar + 8 * (2 * S + 5));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.off_bar + 8 * (2 * S + 5) + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);    // leader's arrive.expect_tx for both CTAs' bytes
            mbar_init(bar_empty + 8 * s, 1);   // leader's MMA commit, multicast to both CTAs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);               // leader's commit after a tile, multicast
            mbar_init(bar_tempty + 8 * b, 2 * EPI_WARPS);  // epilogue warps of both CTAs (leader's copy is used)
        }
        mbar_init(bar_drain, 1);               // leader's final commit, multicast
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmM);
        tma_prefetch_desc(&tmN1);
        if (p.n2) tma_prefetch_desc(&tmN2);
        tma_prefetch_desc(&tmSFM);
        tma_prefetch_desc(&tmSFN);
        if (p.tma_store) tma_prefetch_desc(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // everything below reads the plan and scale blocks of the preceding kernel
    griddep_wait();

    // mode 1: the number of row tiles depends on the routing; the plan holds the item count
    const int nt_per_expert = p.tiles_m * p.tiles_n;
    const long long total =
        p.mode == 0 ? static_cast<long long>(p.E) * nt_per_expert : static_cast<long long>(__ldg(p.plan));
    const int G = gridDim.x / 2, pair = blockIdx.x / 2;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            // bytes both CTAs' copies deliver to the leader's full barrier per stage
            const uint32_t pair_tx = 2u * (static_cast<uint32_t>(A_STAGE) + p.b_stage + SF_ATOM + sfb_stage);
            const uint32_t full_leader = mapa_shared(bar_full, 0);
            const int h1 = p.n1 >> 1, h2 = p.n2 >> 1;
            uint32_t c = 0;
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            ItemStream items(p, G, pair, total);
            Item it;
            unsigned int nbar = 0;  // pass barriers met so far
            while (ok && items.next(it)) {
                if (p.pass_bar && pass_barrier_at(items.cur / G, G, total, nt_per_expert)) {
                    // Pass q starts together on every pair after a pass that held
                    // two experts' tiles (of different lengths): pairs that share
                    // an expert's operands then stream them at the same time and
                    // meet in L2 instead of re-reading them from DRAM. Every CTA
                    // of the grid is resident (the grid is the resident pairs),
                    // every CTA has exactly one item in a full pass, and the wait
                    // is bounded (an abort elsewhere ends it as a timeout here).
                    ++nbar;
                    ok = pass_barrier_wait(p.pass_ctr, nbar * gridDim.x, abort_flag, p.wait_ns);
                    if (!ok) break;
                }
                const int m_row = it.m0 + static_cast<int>(rank) * BM;
                const int n_row1 = it.tn * p.tn + static_cast<int>(rank) * h1;
                const int n_row2 = it.tn * p.tn + p.n1 + static_cast<int>(rank) * h2;
                const int sfm_row = it.sfm + static_cast<int>(rank);
                const int sfn_row = it.sfn;
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    // test hook: only the (over-declared) first fill is issued, so the
                    // stuck phase is never re-armed
                    if (p.stall_first_stage && c >= 1) { ok = false; break; }
                    if (!wait_phase(bar_empty + 8 * st, ph ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
                    const uint32_t fb = full_leader + 8 * st;
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * st, pair_tx + (p.stall_first_stage ? 16u : 0u));
                    const int x = it.start + s * BK;
                    const uint32_t b_dst = sbase + p.off_b + st * p.b_stage;
                    tma_load_2d_pair(sbase + st * A_STAGE, &tmM, fb, x, m_row);
                    tma_load_3d_pair(b_dst, &tmN1, fb, x, n_row1, it.z);
                    if (h2) tma_load_3d_pair(b_dst + h1 * BK, &tmN2, fb, x, n_row2, it.z);
                    tma_load_2d_pair(sbase + p.off_sfa + st * SF_ATOM, &tmSFM, fb, 0, sfm_row + 2 * s);
                    tma_load_2d_pair(sbase + p.off_sfb + st * sfb_stage, &tmSFN, fb, 0, sfn_row + p.nblk_n * s);
                    if (++st == S) { st = 0; ph ^= 1; }
                }
            }
            if (leader && (!ok || *abort_flag)) {
                // let every copy still in flight land before the pair exits
                const uint32_t n = c < static_cast<uint32_t>(S) ? c : static_cast<uint32_t>(S);
                for (uint32_t d = 1; d <= n; ++d) {
                    const uint32_t j = c - d;
                    drain_phase(bar_full + 8 * (j % S), (j / S) & 1, p.wait_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only; see mma_issue)
        if (leader) {
            const MmaCtx ctx{tmem, sbase, bar_empty, bar_tfull, bar_tempty, bar_drain, abort_flag, lane, G, pair, total,
                             nt_per_expert};
            switch (p.nblk_n) {
                case 1: mma_issue<1>(p, ctx); break;
                case 2: mma_issue<2>(p, ctx); break;
                case 3: mma_issue<3>(p, ctx); break;
                default: mma_issue<4>(p, ctx); break;
            }
        }
        if (lane == 0) drain_phase(bar_drain, 0, p.wait_ns);
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ stage watcher (leader only)
        // Waits (bounded) for each stage's data and hands it to the MMA warp
        // through BAR_READY; after an abort it stops waiting but keeps the
        // barrier pairing until the schedule ends. With fewer scale-factor
        // slots than stages it also waits until the MMAs that last read the
        // step's slot (sf_slots steps back) have completed, before the MMA
        // warp copies new scales into it.
        if (leader) {
            uint32_t c = 0;
            bool live = true;
            const bool gate = p.sf_slots < S;
            ItemStream items(p, G, pair, total);
            Item it;
            while (items.next(it)) {
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const uint32_t st = c % S;
                    if (c >= static_cast<uint32_t>(S)) named_bar_sync(BAR_FREE + st, 64);  // MMA warp took the previous fill
                    if (live) {
                        bool ok = true;
                        if (lane == 0) {
                            ok = wait_phase(bar_full + 8 * st, (c / S) & 1, abort_flag, p.wait_ns);
                            if (ok && gate && c >= static_cast<uint32_t>(p.sf_slots)) {
                                const uint32_t j = c - p.sf_slots;
                                ok = wait_phase(bar_empty + 8 * (j % S), (j / S) & 1, abort_flag, p.wait_ns);
                            }
                        }
                        live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    }
                    named_bar_arrive(BAR_READY + st, 64);
                }
            }
            // consume the MMA warp's last BAR_FREE arrivals so every id ends paired
            for (uint32_t d = c < static_cast<uint32_t>(S) ? c : static_cast<uint32_t>(S); d > 0; --d)
                named_bar_sync(BAR_FREE + (c - d) % S, 64);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (8 warps per CTA)
        // TMEM lane = M-side row of this CTA's half, column = N-side row of the
        // tile. Two warps share each 32-lane quarter, each draining half of the
        // tn columns (at most 224) in 32-column chunks. Up to four chunks are
        // loaded together, the accumulator is released, then they are stored.
        // Five to seven chunks (32-byte or TMA stores): a seventh is loaded and
        // stored first, then chunks 0-5 are narrowed to bf16 pairs as each
        // lands (96 registers), the accumulator is released and they are
        // stored. With 16-byte stores, batches of at most four chunks (fp32
        // registers hold 128 columns at most), the short one first, the
        // release after the last batch's loads.
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int h = (warp - EPI_WARP0) >> 2;  // column half of the tile
        const int ncols = p.tn >> 1;
        const int nchunks = (ncols + 31) >> 5;
        const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
        // the loop is instantiated per accumulator count (1 or 2), which keeps
        // the buffer index out of the registers the TMEM loads need
        auto epilogue_loop = [&](auto nbuf_tag, auto mode_tag, auto packed_tag) {
            constexpr uint32_t BUF_SHIFT = decltype(nbuf_tag)::value == 2 ? 1u : 0u;
            // the drained row held as bf16 pairs (five to seven chunks; a
            // seventh is stored before the others are loaded)
            constexpr bool PACKED = decltype(packed_tag)::value != 0;
            constexpr int PACK_CHUNKS = 6;
            // 0: the M side on the output's rows (rows of A, or of X in the
            // grouped GEMM), 16-byte stores; 1: the same with 32-byte stores;
            // 2: the M side on the output's columns (rows of B; transposed:
            // 4-byte stores, or TMA stores through shared memory when
            // p.tma_store); 3: as 0, through shared memory and TMA stores
            constexpr int MODE = decltype(mode_tag)::value;
            uint32_t ntile = 0;  // non-empty tiles drained so far
            // MODE 3: this warp's staging buffers (2 KB each) and the next one to fill
            const uint32_t stg_warp =
                sbase + p.off_stg + static_cast<uint32_t>((warp - EPI_WARP0) * p.stg_bufs) * STG_CHUNK;
            uint32_t sbuf = 0;
            const bool odd = lane & 1;
            // (no look-ahead here: the item's loads overlap the wait for its
            // accumulator; 32-bit counters: the item count is below 2^31)
            const int total32 = static_cast<int>(total);
            for (int pass = 0; pass * G < total32; ++pass) {
                const int i = (pass & 1) ? pass * G + (G - 1 - pair) : pass * G + pair;
                if (i >= total32) continue;
                const Item it = load_item(p, i);
                const int mrow = it.m0 + static_cast<int>(rank) * BM + q * 32 + lane;  // this lane's M-side row
                const int ncol0 = it.tn * p.tn + h * ncols;                                      // first N-side row here
                // NK: a lane owns output row mrow; KN: a lane owns output column
                // mrow, and lane pairs share the column pair (k2, k2 + 1)
                const int k2 = mrow & ~1;
                const bool row_in = MODE == 2 ? (k2 < p.K) : (mrow < it.m_end);
                uint16_t* obase = MODE == 2 ? p.out + static_cast<size_t>(it.g) * p.N * static_cast<size_t>(p.K) + k2
                                       : p.out + static_cast<size_t>(it.orow0 + mrow) * static_cast<size_t>(p.out_stride) + ncol0;
                // Narrow one 32-column chunk (columns 32 j .. 32 j + 31 of this warp's
                // half) to bf16 and store it. NK: 16-byte runs of the lane's row.
                // KN: neighbouring lanes swap their (n, n+1) pairs so that the even
                // lane stores (k, k+1) of row n and the odd lane (k, k+1) of row
                // n+1: 4-byte stores, 64 contiguous bytes per row and instruction.
                // w(i) gives columns 2i and 2i + 1 of the chunk as a bf16 pair.
                auto store_chunk = [&](int j, auto w) {
                    if (MODE == 2 && p.tma_store) {
                        // transposed tile through a staging buffer: the chunk is
                        // output rows n = ncol0 + 32 j .. + 31 (TMEM columns) by
                        // columns k = the warp's 32 lanes; after the pair exchange
                        // below, the even lane holds (k, k + 1) of row n and the odd
                        // lane those of row n + 1. Staged as 32 rows (n) x 64 bytes
                        // with the 64-byte swizzle: one 4-byte store per lane and
                        // column pair, rows n and n + 1 in different bank halves
                        const int k0w = it.m0 + static_cast<int>(rank) * BM + q * 32;
                        if (32 * j + 32 <= ncols && k0w < p.K && ncol0 + 32 * j < p.N) {
                            if (lane == 0) {
                                if (p.stg_bufs == 2) bulk_wait_group_read<1>();
                                else bulk_wait_group_read<0>();
                            }
                            __syncwarp();
                            const uint32_t buf = stg_warp + sbuf * STG_CHUNK;
                            const uint32_t kb = static_cast<uint32_t>(lane & ~1) * 2u;  // byte of k2 in the row
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                const uint32_t mine = w(c >> 1);
                                const uint32_t got = __shfl_xor_sync(0xffffffffu, mine, 1);
                                const uint32_t x =
                                    odd ? __byte_perm(got, mine, 0x7632) : __byte_perm(mine, got, 0x5410);
                                const uint32_t r = static_cast<uint32_t>(c) + (odd ? 1u : 0u);
                                const uint32_t piece = (kb >> 4) ^ ((r >> 1) & 3u);
                                st_shared_b32(buf + r * 64u + piece * 16u + (kb & 15u), x);
                            }
                            fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&tmOut, buf, k0w, ncol0 + 32 * j, it.g);
                                bulk_commit_group();
                            }
                            sbuf ^= static_cast<uint32_t>(p.stg_bufs - 1);
                            return;
                        }
                        // a partial chunk: the 4-byte stores below
                    }
                    if (MODE == 3) {
                        // whole 32 x 32 chunks (inside this warp's columns and, for
                        // ragged rows, inside the group) go through a staging buffer:
                        // lane = row, 64 bytes per row, 16-byte pieces placed by the
                        // 64-byte swizzle (piece ^ bits 7-8 of the address), which
                        // keeps the shared stores conflict-free; the TMA store
                        // clips rows and columns outside the output
                        const int row0w = it.m0 + static_cast<int>(rank) * BM + q * 32;
                        // (a chunk that starts outside the output has nothing to store: the
                        // checks of the 16-byte path below skip all of it)
                        if (32 * j + 32 <= ncols && row0w < it.m_end && ncol0 + 32 * j < p.col_limit &&
                            (p.mode == 0 || row0w + 32 <= it.m_end)) {
                            if (lane == 0) {
                                if (p.stg_bufs == 2) bulk_wait_group_read<1>();
                                else bulk_wait_group_read<0>();
                            }
                            __syncwarp();
                            const uint32_t buf = stg_warp + sbuf * STG_CHUNK;
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const uint32_t piece = static_cast<uint32_t>(c4) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u);
                                st_shared_v4(buf + static_cast<uint32_t>(lane) * 64u + piece * 16u,
                                             w(4 * c4 + 0), w(4 * c4 + 1), w(4 * c4 + 2), w(4 * c4 + 3));
                            }
                            fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&tmOut, buf, ncol0 + 32 * j, row0w, p.mode == 0 ? it.g : 0);
                                bulk_commit_group();
                            }
                            sbuf ^= static_cast<uint32_t>(p.stg_bufs - 1);
                            return;
                        }
                        // partial chunks: the 16-byte stores below
                    }
                    if (MODE == 1) {
                        // one full 32-byte sector per lane and store
#pragma unroll
                        for (int c = 0; c < 32; c += 16) {
                            const int cc = 32 * j + c;
                            if (row_in && cc < ncols && ncol0 + cc < p.col_limit)
                                st_global_v8(obase + cc, w(c / 2 + 0), w(c / 2 + 1), w(c / 2 + 2), w(c / 2 + 3),
                                             w(c / 2 + 4), w(c / 2 + 5), w(c / 2 + 6), w(c / 2 + 7));
                        }
                    } else if (MODE == 0 || MODE == 3) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            const int cc = 32 * j + c;
                            if (row_in && cc < ncols && ncol0 + cc < p.col_limit)
                                *reinterpret_cast<uint4*>(obase + cc) =
                                    make_uint4(w(c / 2 + 0), w(c / 2 + 1), w(c / 2 + 2), w(c / 2 + 3));
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const int cc = 32 * j + c;
                            if (cc < ncols) {  // the same for the whole warp
                                const uint32_t mine = w(c >> 1);
                                const uint32_t got = __shfl_xor_sync(0xffffffffu, mine, 1);
                                // even: (own n, partner n) = row n; odd: (partner n+1, own n+1) = row n+1
                                const uint32_t x = odd ? __byte_perm(got, mine, 0x7632) : __byte_perm(mine, got, 0x5410);
                                const int n = ncol0 + cc + (odd ? 1 : 0);
                                if (row_in && n < p.N) *reinterpret_cast<uint32_t*>(obase + static_cast<size_t>(n) * p.K) = x;
                            }
                        }
                    }
                };
                if (it.nsteps == 0) {
                    // expert without tokens: an exact +0.0 tile, no accumulator involved
                    for (int j = 0; j < nchunks; ++j) store_chunk(j, [](int) { return 0u; });
                    continue;
                }
                // one lane waits, the warp follows its verdict (the TMEM loads below
                // are warp-collective, so the lanes must not split on a timeout)
                bool ready = true;
                const uint32_t buf = ntile & BUF_SHIFT, acc_phase = (ntile >> BUF_SHIFT) & 1u;
                if (lane == 0) ready = wait_phase(bar_tfull + 8 * buf, acc_phase, abort_flag, p.wait_ns);
                if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) break;
                tc_fence_after();
                const uint32_t taddr =
                    tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * static_cast<uint32_t>(p.tn) + static_cast<uint32_t>(h * ncols);
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        // this CTA's half of the accumulator may be overwritten
                        if (leader) mbar_arrive(bar_tempty + 8 * buf);
                        else mbar_arrive_cluster(tempty_leader + 8 * buf);
                    }
                };
                if (PACKED) {
                    // five to seven chunks: a seventh is loaded and stored first;
                    // chunks 0-5 are narrowed to bf16 pairs as soon as each is
                    // loaded, so they fit in registers together and the
                    // accumulator is released before they are stored
                    if (nchunks > PACK_CHUNKS) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + 32 * PACK_CHUNKS, v);
                        tmem_wait_ld();
                        reg_fence(v);
                        store_chunk(PACK_CHUNKS, [&](int i) { return pack_bf16x2(v[2 * i], v[2 * i + 1]); });
                    }
                    uint32_t w[PACK_CHUNKS][16];
#pragma unroll
                    for (int j = 0; j < PACK_CHUNKS; ++j) {
                        if (j < nchunks) {  // (always, with a seventh chunk)
                            uint32_t v[32];
                            tmem_ld_32x32b_x32(taddr + 32 * j, v);
                            tmem_wait_ld();
                            reg_fence(v);
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[j][i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                        }
                    }
                    release();
#pragma unroll
                    for (int j = 0; j < PACK_CHUNKS; ++j)
                        if (j < nchunks) store_chunk(j, [&](int i) { return w[j][i]; });
                } else {
                    // batches of at most four chunks, the short one first: the
                    // accumulator is released after the last batch's loads, so
                    // only the first batch's stores precede the release
                    const int first = nchunks - 4 * ((nchunks - 1) >> 2);
#pragma unroll 1
                    for (int j0 = 0, nb = first; j0 < nchunks; j0 += nb, nb = 4) {
                        uint32_t v[4][32];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j < nb) tmem_ld_32x32b_x32(taddr + 32 * (j0 + j), v[j]);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j) reg_fence(v[j]);
                        if (j0 + nb >= nchunks) release();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (j < nb)
                                store_chunk(j0 + j, [&](int i) { return pack_bf16x2(v[j][2 * i], v[j][2 * i + 1]); });
                        }
                    }
                }
                ++ntile;
            }
            if (MODE == 3 || (MODE == 2 && p.tma_store)) {
                // every TMA store of this warp has completed before the CTA may exit
                if (lane == 0) bulk_wait_group_all();
                __syncwarp();
            }
        };
        using I1 = std::integral_constant<int, 1>;
        using I2 = std::integral_constant<int, 2>;
        using I0 = std::integral_constant<int, 0>;
        using I3 = std::integral_constant<int, 3>;
        const int mode = p.kn ? 2 : (p.tma_store ? 3 : (p.wide_stores ? 1 : 0));
        // (two accumulators only where tn <= 224: at most four chunks per warp)
        const bool packed = p.acc_bufs == 1 && nchunks > 4 && mode != 0;
        switch ((p.acc_bufs == 2 ? 4 : 0) + mode + (packed ? 8 : 0)) {
            case 0: epilogue_loop(I1{}, I0{}, I0{}); break;
            case 1: epilogue_loop(I1{}, I1{}, I0{}); break;
            case 2: epilogue_loop(I1{}, I2{}, I0{}); break;
            case 3: epilogue_loop(I1{}, I3{}, I0{}); break;
            case 4: epilogue_loop(I2{}, I0{}, I0{}); break;
            case 5: epilogue_loop(I2{}, I1{}, I0{}); break;
            case 6: epilogue_loop(I2{}, I2{}, I0{}); break;
            case 9: epilogue_loop(I1{}, I1{}, I1{}); break;
            case 10: epilogue_loop(I1{}, I2{}, I1{}); break;
            case 11: epilogue_loop(I1{}, I3{}, I1{}); break;
            default: epilogue_loop(I2{}, I3{}, I0{}); break;
        }
    }

    // both CTAs stay resident until the pair's MMAs, copies and TMEM reads are
    // done, then free the pair's TMEM together
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

// ============================================================== host side

namespace {

// Shared-memory and TMEM geometry of the main kernel for an N-side tile of
// tn rows; false if it does not fit.
struct Geometry {
    int stages, sf_slots, acc_bufs;
    int stg_bufs;  // TMA-store staging buffers per epilogue warp (0: none fit)
    uint32_t sf_col0;
    uint32_t off_b, off_sfa, off_sfb, off_stg, off_bar, b_stage, smem_bytes;
};

// TMEM: one or two accumulators of tn columns, then the scale-factor slots.
// Two accumulators when they fit beside one slot per stage (tn <= 224 with
// 6-7 stages), else one with as many slots as fit (at least 2). Shared
// memory: as many operand stages as fit (each one measured worth 5-8% at
// 4-5 stages), then, only in what is left, one or two 2 KB staging buffers per
// epilogue warp for the TMA-store epilogue.
bool geometry(int tn, Geometry* g) {
    const int nblk = (tn + 127) / 128;
    const uint32_t b_stage = static_cast<uint32_t>(tn / 2) * BK;  // multiple of 1024 (tn % 16 == 0)
    const uint32_t per_stage = A_STAGE + b_stage + SF_ATOM + nblk * SF_ATOM + 16;  // + two mbarriers
    const uint32_t fixed = 1024 + 5 * 8 + 16;  // alignment slack, tile barriers, abort flag / TMEM slot
    int stages = static_cast<int>((MAIN_SMEM_MAX - fixed) / per_stage);
    if (stages > MAX_STAGES) stages = MAX_STAGES;
    const int sf_cols = 4 + 4 * nblk;
    int bufs = (2 * tn + stages * sf_cols <= static_cast<int>(TMEM_COLS)) ? 2 : 1;
    int slots = (static_cast<int>(TMEM_COLS) - bufs * tn) / sf_cols;
    if (slots > stages) slots = stages;
    if (stages < 3 || slots < 2) return false;
    g->stages = stages;
    g->sf_slots = slots;
    g->acc_bufs = bufs;
    g->sf_col0 = static_cast<uint32_t>(bufs * tn);
    g->b_stage = b_stage;
    g->off_b = static_cast<uint32_t>(stages) * A_STAGE;
    g->off_sfa = g->off_b + stages * b_stage;
    g->off_sfb = g->off_sfa + stages * SF_ATOM;
    const uint32_t sf_end = g->off_sfb + stages * nblk * SF_ATOM;
    const uint32_t bars = 8 * (2 * stages + 5) + 16 + 1024;  // barriers, flag, TMEM slot, base alignment slack
    g->off_stg = (sf_end + 1023u) & ~1023u;
    g->stg_bufs = 0;
    for (int nb = 2; nb >= 1; --nb)
        if (g->off_stg + nb * EPI_WARPS * STG_CHUNK + bars <= static_cast<uint32_t>(MAIN_SMEM_MAX)) {
            g->stg_bufs = nb;
            break;
        }
    g->off_bar = g->stg_bufs ? g->off_stg + g->stg_bufs * EPI_WARPS * STG_CHUNK : sf_end;
    g->smem_bytes = g->off_bar + bars;
    return g->smem_bytes <= static_cast<uint32_t>(MAIN_SMEM_MAX);
}

// Relative time per computed output column of one pair K-step with an
// N-side tile of tn rows, measured with this kernel on GB300 under its power
// cap (whole-kernel time / (tiles x tn), normalised to tn = 256, on the 671B
// up/gate and down expert shapes with the 256 side on A). Narrow tiles pay the
// per-step scale-factor copies and the M-side operand bytes over fewer
// columns; tn just above 256 adds a second MMA too narrow to run at full
// rate; around 384-448 the operand bytes per column are lowest. The entry
// for 352 comes from the 16B expert shape instead (tn = 352 against 416 with
// the 256 side on A, at 4096 and 24576 tokens per expert: 0.917-0.92).
double column_cost(int tn) {
    static const double f[] = {
        // tn = 16, 32, ..., 448
        3.00, 2.60, 2.30, 2.00, 1.85, 1.70, 1.60, 1.49,         // 16 .. 128
        1.28, 1.175, 1.14, 1.063, 1.063, 1.002, 0.985, 1.00,    // 144 .. 256
        1.094, 1.039, 1.066, 1.023, 0.982, 0.92, 0.948, 0.914,  // 272 .. 384
        0.919, 0.89, 0.912, 0.902};                             // 400 .. 448
    return f[tn / 16 - 1];
}

TileConfig make_config(int kn, int tn, int rows_m, int rows_n) {
    TileConfig tc;
    tc.kn = kn;
    tc.tn = tn;
    tc.n1 = tn < 256 ? tn : 256;
    tc.n2 = tn - tc.n1;
    tc.nblk_n = (tn + 127) / 128;
    tc.tiles_m = (rows_m + PAIR_M - 1) / PAIR_M;
    tc.tiles_n = (rows_n + tn - 1) / tn;
    tc.m_fastest = MXW_ORDER >= 0 ? MXW_ORDER : (rows_m < rows_n ? 1 : 0);
    return tc;
}

// Best tile of one orientation: the modelled time of all tiles of an expert
// of `steps` K-steps over every admissible tn; ties keep the larger tn. In
// units of one K-step of one output column at tn = 256, a tile costs
//   max(steps x tn x column_cost(tn), W x tn) + 205,
// measured on GB300: the column costs include the tile hand-overs at 65-130
// K-steps per tile, plus three K-steps when a one-accumulator tile is wider
// than 256 (its epilogue stores half of its columns before loading the
// rest); W is the output-write floor of a short tile (its 256 x tn bf16
// stores: about 6.6 K-steps with 32-byte stores, 13 with 16-byte ones, 17 for
// the transposed 4-byte stores of the 256 side on B), 205 a fixed per-tile
// cost; widths whose TMA-store staging fits and whose chunks are all staged
// (tn % 64 == 0) have the floor 3.7 tn + 815 instead. The 256 side on B also
// measured, weighed with the column costs above, about 8% slower on long
// tiles with its 4-byte register stores; about 4% slower where its chunks go
// through TMA stores but half a chunk still leaves from registers (tn % 64 ==
// 32: 8 x 4 tiles of 352 on B against 6 x 5 of 416 on A at the 16B expert
// shape; 28 x 10 tiles of 416 on B ran 8% slower than 16 x 16 of 448 on A at
// the 671B up/gate shape); and about 1% faster where every chunk is staged
// (tn % 64 == 0: 16 x 8 tiles of 448 on B ran 1.8% faster than 28 x 5 of 416
// on A at the 671B down shape, main kernel, four interleaved pairs of runs).
TileConfig best_of(int kn, int rows_m, int rows_n, double steps, int force_tn, bool wide_ok, double* cost) {
    TileConfig best{};
    double best_cost = -1.0;
    for (int tn = MAX_TN; tn >= 16; tn -= 16) {
        if (force_tn && tn != force_tn) continue;
        Geometry g;
        if (!geometry(tn, &g)) continue;
        const TileConfig tc = make_config(kn, tn, rows_m, rows_n);
        const bool wide = !kn && wide_ok && tn % 32 == 0;
        const double w_floor = kn ? 17.0 : (wide ? 6.6 : 13.0);
        const double kn_factor = g.stg_bufs == 0 ? 1.08 : (tn % 64 == 0 ? 0.99 : 1.04);
        const double run = (steps + (g.acc_bufs == 1 && tn > 256 ? 3.0 : 0.0)) * tn * column_cost(tn) * (kn ? kn_factor : 1.0);
        double per_tile = (run > w_floor * tn ? run : w_floor * tn) + 205.0;
        if (!kn && g.stg_bufs > 0 && tn % 64 == 0) {
            // TMA-store epilogue with every 32-column chunk staged: a short tile
            // is bound by 3.7 K-steps per column plus a fixed 815 (measured at
            // 1-2 K-steps per tile, E = 160 and 512)
            const double floor_tma = 3.7 * tn + 815.0;
            per_tile = run + 205.0 > floor_tma ? run + 205.0 : floor_tma;
        }
        const double c = static_cast<double>(tc.tiles_m) * tc.tiles_n * per_tile;
        if (best_cost < 0 || c < best_cost * (1.0 - 1e-9)) {
            best_cost = c;
            best = tc;
        }
    }
    *cost = best_cost;
    return best;
}

// Whether the weight gradient's producers should meet at expert boundaries
// (pass_barrier_at). A pass of the G pairs covers G consecutive tiles; the
// operand indexed by the faster-moving tile index is shared by the pairs
// `inner` apart in a pass (G / inner of them), and pairs that start their
// tiles at different times stream it at different times, so the L2 no longer
// serves them all and it is re-read from DRAM (measured at 671B down:
// 11-18 GB read per launch against 5 GB of operands, 7.2 GB with the
// barrier). The barrier costs the idle time of the pairs that finish a pass
// early, small only when a pass mostly holds one expert. Measured on GB300
// with one call per variant: 671B down on 28 x 5 tiles of 416 (140 tiles per
// expert, 15 pairs sharing each N-side tile) +2.6% back to back; 671B down on
// 16 x 8 tiles of 448 with the 256 side on B (128 tiles, 9.5 pairs sharing
// each stripe of A) DRAM reads 7.4 -> 7.0 GB, main kernel +2.5% after L2
// flushes and -1.2% back to back (two interleaved pairs of runs); 671B
// up/gate (256 tiles, 4.75 pairs sharing each M-side stripe) -1%; 16B and
// 16B production (32 tiles per expert, two or three experts per pass) -6%
// and -2.5%. On: at least one pass of tiles per expert and at least 8 pairs
// sharing each far tile.
int use_pass_barrier(const TileConfig& tc, int G) {
    const long long ntpe = static_cast<long long>(tc.tiles_m) * tc.tiles_n;
    const int inner = tc.m_fastest ? tc.tiles_m : tc.tiles_n;
    return (ntpe >= G && G >= 8 * inner) ? 1 : 0;
}

static cudaError_t launch_main(MainParams& mp, const TileConfig& tc, const Geometry& geo, long long items,
                               const CUtensorMap* maps, int dev, int num_sms, cudaStream_t stream,
                               cudaEvent_t ev_before, cudaEvent_t ev_after);

}  // namespace

bool choose_tiles(int N, int K, int E, int64_t M, int force, int force_tn, TileConfig* tc) {
    if (N < 1 || K < 1) return false;
    if (force_tn && (force_tn < 16 || force_tn > MAX_TN || force_tn % 16)) return false;
    const double steps = (E > 0 && M > 0) ? static_cast<double>(M) / (static_cast<double>(E) * BK) + 1.0 : 32.0;
    double c_nk, c_kn;
    // 32-byte output stores need 16-column-aligned output rows (K % 16 == 0)
    const TileConfig nk = best_of(0, N, K, steps, force_tn, K % 16 == 0, &c_nk);
    const TileConfig kn = best_of(1, K, N, steps, force_tn, K % 16 == 0, &c_kn);
    if (c_nk < 0 || c_kn < 0) return false;
    if (force == 1) *tc = nk;
    else if (force == 2) *tc = kn;
    else *tc = c_kn < c_nk * (1.0 - 1e-9) ? kn : nk;  // ties keep the row-contiguous epilogue
    return true;
}

bool ws_layout(int E, int N, int K, int64_t M, const TileConfig& tc, WsLayout* L) {
    if (E < 1 || E > MXFP8_MAX_EXPERTS || N < 1 || K < 1 || M < 32 || (M % 32) != 0) return false;
    if (M > (int64_t(1) << 31) - 256) return false;
    const int64_t ts = (M + BK - 1) / BK + E;
    // scale-factor block rows (tile * ts_max + step) * blocks + block are int32 TMA coordinates
    const int64_t rows_m = static_cast<int64_t>(tc.tiles_m) * ts * 2;
    const int64_t rows_n = static_cast<int64_t>(tc.tiles_n) * ts * tc.nblk_n;
    if (rows_m > (int64_t(1) << 31) - 1 || rows_n > (int64_t(1) << 31) - 1) return false;
    // work items (expert, tile) are counted in 32-bit integers in the kernel
    if (static_cast<int64_t>(E) * tc.tiles_m * tc.tiles_n > (int64_t(1) << 31) - 1) return false;
    L->ts_max = static_cast<int>(ts);
    L->tc = tc;
    const size_t plan_bytes = sizeof(int32_t) * (PLAN_HDR + 5 * static_cast<size_t>(E));
    L->plan_off = 0;
    L->sfm_off = (plan_bytes + 1023) & ~size_t(1023);
    L->sfn_off = L->sfm_off + static_cast<size_t>(rows_m) * SF_ATOM;
    L->total = L->sfn_off + static_cast<size_t>(rows_n) * SF_ATOM;
    return true;
}

size_t ws_bytes_any_orientation(int E, int N, int K, int64_t M, int force_tn) {
    size_t most = 0;
    for (int force = 1; force <= 2; ++force) {
        TileConfig tc;
        WsLayout L;
        if (!choose_tiles(N, K, E, M, force, force_tn, &tc) || !ws_layout(E, N, K, M, tc, &L)) return 0;
        if (L.total > most) most = L.total;
    }
    return most;
}

cudaError_t load_kernel_modules() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, wgrad_prep);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, wgrad_main);
    return e;
}

cudaError_t launch_wgrad(const WgradArgs& a, const CUtensorMap* maps, const char** what) {
    const WsLayout& L = a.lay;
    const TileConfig& tc = L.tc;
    int32_t* plan = reinterpret_cast<int32_t*>(a.ws + L.plan_off);
    Geometry geo;
    *what = "tile geometry";
    if (!geometry(tc.tn, &geo)) return cudaErrorInvalidConfiguration;

    *what = "plan / scale re-layout kernel";
    {
        PrepSide sm_side, sn_side;
        sm_side.plane = tc.kn ? a.sB : a.sA;
        sm_side.rows = tc.kn ? a.K : a.N;
        sm_side.tile_rows = PAIR_M;
        sm_side.tiles = tc.tiles_m;
        sm_side.blocks = 2;
        sm_side.sf = a.ws + L.sfm_off;
        sn_side.plane = tc.kn ? a.sA : a.sB;
        sn_side.rows = tc.kn ? a.N : a.K;
        sn_side.tile_rows = tc.tn;
        sn_side.tiles = tc.tiles_n;
        sn_side.blocks = tc.nblk_n;
        sn_side.sf = a.ws + L.sfn_off;
        if (!a.gather) {
            // the caller's scale-factor blocks: the prep only writes the plan
            sm_side.rows = sn_side.rows = 0;
            sm_side.tiles = sn_side.tiles = 0;
        }
        // enough blocks for every task of the largest possible plan, at most as
        // many as are resident at once (one wave)
        const long long tasks = (2LL * sm_side.tiles + static_cast<long long>(tc.nblk_n) * sn_side.tiles) *
                                ((L.ts_max + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS);
        const size_t sm = sizeof(int) * (3 * static_cast<size_t>(a.E) + 1) +
                          sizeof(uint32_t) * PREP_ROWS * (PREP_TILE_STEPS + 1);
        // (large E can need more than the 48 KB default of shared memory)
        // (per-device caches below: idempotent, so concurrent first calls may
        // both set them; atomics keep that free of data races)
        static std::atomic<bool> prep_attr[64];
        if (a.dev < 0 || a.dev >= 64) return cudaErrorInvalidDevice;
        if (!prep_attr[a.dev].load(std::memory_order_relaxed)) {
            cudaError_t e0 = cudaFuncSetAttribute(wgrad_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
            if (e0 != cudaSuccess) return e0;
            prep_attr[a.dev].store(true, std::memory_order_relaxed);
        }
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wgrad_prep, PREP_THREADS, sm);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        long long blocks = tasks + (a.grid ? 1 : 0);  // on the grid block 0 only plans
        if (blocks > static_cast<long long>(per_sm) * a.num_sms) blocks = static_cast<long long>(per_sm) * a.num_sms;
        if (blocks < 1) blocks = 1;
        // The L2 prefetch of the planes at the prep's entry pays while its
        // gather waits for offs, or while the planes fit well within L2 (16B:
        // the flushed step 2% faster with it); on the grid with planes of
        // 90-150 MB (the 671B shapes) the prefetched lines are evicted before
        // the gather reaches them (671B down: 236 MB read instead of 151,
        // 72 instead of 62 us).
        const size_t plane_bytes = (static_cast<size_t>(sm_side.rows) + sn_side.rows) * static_cast<size_t>(a.M / 32);
        const int prefetch = (!a.grid || plane_bytes <= (size_t(64) << 20)) ? 1 : 0;
        wgrad_prep<<<static_cast<unsigned>(blocks), PREP_THREADS, sm, a.stream>>>(a.offs, sm_side, sn_side, plan, a.E,
                                                                                    a.M, L.ts_max, a.grid, prefetch);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    *what = "main contraction kernel";
    MainParams mp;
    mp.plan = plan;
    mp.out = a.out;
    mp.mode = 0;
    mp.grid = a.grid;
    mp.pass_ctr = reinterpret_cast<unsigned int*>(plan + 2);  // (pass_bar: set in launch_main)
    mp.out_stride = a.K;
    mp.col_limit = a.K;
    mp.ksteps = 0;
    mp.E = a.E;
    mp.N = a.N;
    mp.K = a.K;
    mp.ts_max = L.ts_max;
    mp.tiles_m = tc.tiles_m;
    mp.tma_store = a.tma_store;
    mp.wide_stores = (!tc.kn && tc.tn % 32 == 0 && a.K % 16 == 0 && (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0) ? 1 : 0;
    mp.wait_ns = a.wait_limit_ns;
    mp.stall_first_stage = a.stall_first_stage;
    const long long total = static_cast<long long>(a.E) * tc.tiles_m * tc.tiles_n;
    return launch_main(mp, tc, geo, total, maps, a.dev, a.num_sms, a.stream, a.ev_before, a.ev_after);
}

// The persistent CTA-pair kernel for either mode, as a programmatic
// dependent of the prep kernel just enqueued. `items` bounds the work items
// (the grid is the smaller of it and the resident pairs).
namespace {
cudaError_t launch_main(MainParams& mp, const TileConfig& tc, const Geometry& geo, long long items,
                        const CUtensorMap* maps, int dev, int num_sms, cudaStream_t stream, cudaEvent_t ev_before,
                        cudaEvent_t ev_after) {
    // per device: the shared-memory opt-in and the number of CTA pairs that
    // can be resident at once (the persistent grid; one CTA per SM whatever
    // the tile, as the register file holds only one)
    static std::atomic<int> max_pairs[64];
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int mp_dev = max_pairs[dev].load(std::memory_order_relaxed);
    if (mp_dev == 0) {
        cudaError_t e = cudaFuncSetAttribute(wgrad_main, cudaFuncAttributeMaxDynamicSharedMemorySize, MAIN_SMEM_MAX);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * (num_sms / 2));
        q.blockDim = dim3(MAIN_THREADS);
        q.dynamicSmemBytes = MAIN_SMEM_MAX;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, wgrad_main, &q);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        max_pairs[dev].store(clusters, std::memory_order_relaxed);
        mp_dev = clusters;
    }
    mp.tiles_n = tc.tiles_n;
    mp.tn = tc.tn;
    mp.n1 = tc.n1;
    mp.n2 = tc.n2;
    mp.nblk_n = tc.nblk_n;
    mp.kn = tc.kn;
    mp.m_fastest = mp.mode == 0 ? tc.m_fastest : 0;
    mp.stages = geo.stages;
    mp.sf_slots = geo.sf_slots;
    mp.acc_bufs = geo.acc_bufs;
    mp.sf_col0 = geo.sf_col0;
    mp.off_b = geo.off_b;
    mp.off_sfa = geo.off_sfa;
    mp.off_sfb = geo.off_sfb;
    mp.off_bar = geo.off_bar;
    mp.off_stg = geo.off_stg;
    mp.stg_bufs = geo.stg_bufs;
    // the caller asks for TMA stores (output map built); they run where staging fits
    mp.tma_store = (mp.tma_store && geo.stg_bufs > 0 && (!tc.kn || mp.mode == 0)) ? 1 : 0;
    mp.b_stage = geo.b_stage;
    const int pairs = static_cast<int>(items < mp_dev ? (items > 0 ? items : 1) : mp_dev);
    if (mp.mode == 0) mp.pass_bar = MXW_PASS_BARRIER >= 0 ? MXW_PASS_BARRIER : use_pass_barrier(tc, pairs);
    if (ev_before) {
        cudaError_t e = cudaEventRecord(ev_before, stream);
        if (e != cudaSuccess) return e;
    }
    // programmatic dependent launch: the prologue (barriers, TMEM allocation,
    // descriptor prefetch) overlaps the prep kernel's tail; griddepcontrol.wait
    // in the kernel orders every read of the prep kernel's output after it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(MAIN_THREADS);
    cfg.dynamicSmemBytes = geo.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // the pass barrier has CTAs wait on one another: a cooperative launch
    // guarantees that every CTA of the grid is resident at once
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = mp.pass_bar ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, wgrad_main, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], mp);
    if (e != cudaSuccess && mp.pass_bar) {
        // the grid could not be made co-resident (another context holds SMs):
        // run without the barrier, which needs no co-residency
        (void)cudaGetLastError();
        mp.pass_bar = 0;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, wgrad_main, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], mp);
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev_after) {
        e = cudaEventRecord(ev_after, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// ------------------------------------------------------------- grouped GEMM host side

// Measured cost of one tile of the grouped GEMM (row tiles of 256, a short
// contraction of K/128 steps: 11-56 on the expert shapes), in microseconds
// at about 1.9-2.0 GHz: a fixed hand-over part a(tn) and b(tn) per K-step,
// fitted on GB300 over the forward and data-gradient products of the 16B and
// 671B expert layers (tn = 128 .. 448, each with its default epilogue: TMA
// stores where their staging fits beside the operand ring, e.g. tn = 256,
// 352, 448, else 32-byte register stores where tn % 32 == 0). With one
// accumulator every tile waits for the previous tile's TMEM drain, which
// short tiles do not amortise; tn = 256 (one MMA per 32-element chunk, six
// stages, staged stores) measured best on most shapes; widths of 16 mod 32
// store in 16-byte pieces, part of which falls inside that wait. The fixed
// part of tn = 352 was refitted after the epilogue came to release the
// accumulator before its stores (forward and data gradient of the 16B
// layers against tn = 256, per-step part kept).
double gemm_tile_cost(int tn, bool wide_ok, double steps) {
    static const double ab[][2] = {
        // tn = 128, 144, ..., 448
        {1.09, 0.318}, {1.37, 0.316}, {1.25, 0.321}, {1.28, 0.333}, {1.09, 0.341}, {2.30, 0.340},
        {1.82, 0.360}, {1.64, 0.370}, {1.88, 0.346}, {4.72, 0.474}, {3.28, 0.466}, {5.44, 0.471},
        {2.91, 0.473}, {2.63, 0.520}, {1.64, 0.525}, {2.86, 0.546}, {3.36, 0.529}, {5.27, 0.565},
        {3.00, 0.584}, {2.80, 0.598}, {2.25, 0.624}};
    if (tn < 128) {
        // narrower than measured: the long-tile column cost, scaled from tn = 128
        const double b = ab[0][1] * (tn * column_cost(tn)) / (128.0 * column_cost(128));
        return ab[0][0] + b * steps;
    }
    double a = ab[(tn - 128) / 16][0];
    const double b = ab[(tn - 128) / 16][1];
    // output rows not 16-column aligned: no 32-byte stores for any width
    if (!wide_ok && tn % 32 == 0) a = tn > 256 ? (a > 5.0 ? a : 5.0) : a + 0.5;
    return a + b * steps;
}

bool choose_gemm_tiles(int N, int K, int E, int64_t M, int force_tn, TileConfig* tc) {
    if (N < 1 || K < 32 || E < 1 || M < 1) return false;
    if (force_tn && (force_tn < 16 || force_tn > MAX_TN || force_tn % 16)) return false;
    const double steps = static_cast<double>((K + BK - 1) / BK);
    const int rows_m = static_cast<int>(M < (int64_t(1) << 30) ? M : (int64_t(1) << 30));
    const bool wide_ok = N % 16 == 0;
    double best = -1.0;
    for (int tn = MAX_TN; tn >= 16; tn -= 16) {
        if (force_tn && tn != force_tn) continue;
        Geometry g;
        if (!geometry(tn, &g)) continue;
        // the row tiles are the same for every width: cost per row tile
        const double c = static_cast<double>((N + tn - 1) / tn) * gemm_tile_cost(tn, wide_ok, steps);
        if (best < 0 || c < best * (1.0 - 1e-9)) {
            best = c;
            *tc = make_config(0, tn, rows_m, N);
        }
    }
    return best >= 0;
}

bool gemm_layout(int E, int N, int K, int64_t M, const TileConfig& tc, GemmLayout* L) {
    if (E < 1 || E > MXFP8_MAX_EXPERTS || N < 1 || K < 32 || (K % 32) != 0 || M < 1) return false;
    if (M > (int64_t(1) << 31) - 1) return false;
    const int64_t mtiles = (M + 2 * BM - 1) / (2 * BM) + E;
    const int64_t ksteps = (K + BK - 1) / BK;
    if (mtiles * tc.tiles_n > (int64_t(1) << 31) - 1) return false;
    const int64_t rows_m = mtiles * ksteps * 2;
    const int64_t rows_n = static_cast<int64_t>(E) * tc.tiles_n * ksteps * tc.nblk_n;
    if (rows_m > (int64_t(1) << 31) - 1 || rows_n > (int64_t(1) << 31) - 1) return false;
    L->mtiles_max = static_cast<int>(mtiles);
    L->ksteps = static_cast<int>(ksteps);
    L->tc = tc;
    const size_t plan_bytes = sizeof(int32_t) * (PLAN_HDR + 4 * static_cast<size_t>(mtiles));
    L->plan_off = 0;
    L->sfm_off = (plan_bytes + 1023) & ~size_t(1023);
    L->sfn_off = L->sfm_off + static_cast<size_t>(rows_m) * SF_ATOM;
    L->total = L->sfn_off + static_cast<size_t>(rows_n) * SF_ATOM;
    return true;
}

cudaError_t launch_gemm(const GemmArgs& a, const CUtensorMap* maps, const char** what) {
    const GemmLayout& L = a.lay;
    const TileConfig& tc = L.tc;
    int32_t* plan = reinterpret_cast<int32_t*>(a.ws + L.plan_off);
    Geometry geo;
    *what = "tile geometry";
    if (!geometry(tc.tn, &geo)) return cudaErrorInvalidConfiguration;

    *what = "grouped GEMM plan / scale re-layout kernel";
    {
        GemmPrepArgs pa;
        pa.offs = a.offs;
        pa.sX = a.sX;
        pa.sW = a.sW;
        pa.sfm = a.ws + L.sfm_off;
        pa.sfn = a.ws + L.sfn_off;
        pa.plan = plan;
        pa.out = a.out;
        pa.E = a.E;
        pa.N = a.N;
        pa.K = a.K;
        pa.ksteps = L.ksteps;
        pa.tn = tc.tn;
        pa.tiles_n = tc.tiles_n;
        pa.nblk = tc.nblk_n;
        pa.mtiles_max = L.mtiles_max;
        pa.M = a.M;
        const size_t sm = sizeof(int) * (3 * static_cast<size_t>(a.E) + 1) +
                          sizeof(uint32_t) * PREP_ROWS * (PREP_TILE_STEPS + 1);
        static std::atomic<bool> attr_set[64];
        if (a.dev < 0 || a.dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[a.dev].load(std::memory_order_relaxed)) {
            cudaError_t e0 = cudaFuncSetAttribute(gemm_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
            if (e0 != cudaSuccess) return e0;
            attr_set[a.dev].store(true, std::memory_order_relaxed);
        }
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_prep, PREP_THREADS, sm);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        const long long chunks = (L.ksteps + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS;
        const long long tasks = (2LL * L.mtiles_max + static_cast<long long>(a.E) * tc.tiles_n * tc.nblk_n) * chunks;
        long long blocks = tasks;
        if (blocks > static_cast<long long>(per_sm) * a.num_sms) blocks = static_cast<long long>(per_sm) * a.num_sms;
        if (blocks < 1) blocks = 1;
        gemm_prep<<<static_cast<unsigned>(blocks), PREP_THREADS, sm, a.stream>>>(pa);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    *what = "grouped GEMM main kernel";
    MainParams mp;
    mp.plan = plan;
    mp.out = a.out;
    mp.mode = 1;
    mp.out_stride = a.N;
    mp.col_limit = a.N;
    mp.ksteps = L.ksteps;
    mp.E = a.E;
    mp.N = a.N;
    mp.K = a.K;
    mp.ts_max = 0;
    mp.grid = 0;
    mp.pass_bar = 0;
    mp.pass_ctr = nullptr;
    mp.tiles_m = 0;
    mp.tma_store = a.tma_store;
    mp.wide_stores = (tc.tn % 32 == 0 && a.N % 16 == 0 && (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0) ? 1 : 0;
    mp.wait_ns = a.wait_limit_ns;
    mp.stall_first_stage = 0;
    const long long items = static_cast<long long>(L.mtiles_max) * tc.tiles_n;
    return launch_main(mp, tc, geo, items, maps, a.dev, a.num_sms, a.stream, a.ev_before, a.ev_after);
}

cudaError_t set_suspend_hint(uint32_t ns) { return cudaMemcpyToSymbol(g_suspend_ns, &ns, sizeof(ns)); }

cudaError_t read_device_status(int32_t* status, int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
    if (e != cudaSuccess) return e;
    *status = v;
    if (clear) {
        const int z = 0;
        e = cudaMemcpyToSymbol(g_device_status, &z, sizeof(int));
    }
    return e;
}

}  // namespace mxw
