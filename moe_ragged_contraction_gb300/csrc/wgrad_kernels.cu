// Ragged MXFP8 weight-gradient grouped GEMM for sm_103a.
//
// "Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on MI355X":
//   section 1  — dW[g] = dY[g]^T X[g]; offsets cut the contraction (token) axis;
//                A = dY^T [N,M], B = X^T [K,M] token-contiguous E4M3, one E8M0
//                scale per 32 tokens in planes [N,M/32] and [K,M/32];
//   section 4  — one CTA owns an output tile for its whole reduction (no
//                atomics, bit-reproducible);
//   section 5.3 — ragged runs: runtime length, 32-aligned start, empty experts
//                get an explicit zero store, scale reads stay in bounds;
//   section 5.4 — longest-expert-first order shortens the tail;
//   section 5.5 — bf16 narrowing (round to nearest even) in registers;
//   section 5.6 — scales re-laid out once per call before the main loop.
//
// Two kernels per call:
//   wgrad_prep : reads offs, clamps them, builds the schedule (per-expert
//                start / length / K-steps, longest-first order) and gathers
//                the scale bytes of every (128-row block, K-step) into the
//                512-byte tcgen05 scale-factor block layout.
//   wgrad_main : persistent, warp-specialised: warp 0 issues TMA loads of the
//                A/B K-step tiles and bulk copies of their scale blocks into
//                a STAGES-deep shared-memory ring; warp 1 copies scales to
//                TMEM and issues tcgen05.mma kind::mxf8f6f4 block-scaled MMAs
//                into a 128x256 fp32 TMEM accumulator; warps 2-9 drain TMEM,
//                narrow to bf16 and store.
//
// A K-step starts exactly at the group's first token (TMA coordinates need
// only 16-byte alignment, and 32 tokens are 32 bytes), so there is no leading
// partial step; the last step of a group issues only the ceil(rem/32) MMAs
// that cover its tokens, so bytes past the group end (the next expert's, or
// padding that may hold NaN) are loaded but never consumed.
#include "mxw_internal.h"
#include "mxw_ptx.cuh"
#include "../../include/mxfp8_wgrad.h"

namespace mxw {

__device__ int g_device_status = 0;

// ============================================================== prep kernel

constexpr int PREP_THREADS = 256;
constexpr int PREP_ROWS = 128;        // rows of one scale-factor block
constexpr int PREP_TILE_STEPS = 32;   // K-steps per gather task (one per lane)

// Every block first rebuilds the per-expert runs from offs (one warp, shuffle
// scans; 3E + 1 words of shared memory). Block 0 also writes the plan. Then
// the blocks stride over gather tasks (below), writing the 512-byte
// scale-factor blocks, where row r, 32-token block kb sits at byte
// (r % 32) * 16 + (r / 32) * 4 + kb. Row blocks: A's ceil(N/128) first, then
// B's, two per 256-row B tile.
__global__ void __launch_bounds__(PREP_THREADS) wgrad_prep(const int32_t* __restrict__ offs,
                                                           const uint8_t* __restrict__ sA,
                                                           const uint8_t* __restrict__ sB,
                                                           int32_t* __restrict__ plan, uint8_t* __restrict__ sfa,
                                                           uint8_t* __restrict__ sfb, int E, int N, int K,
                                                           long long M, int ts_max, int ntn, int ntk) {
    extern __shared__ int prep_smem[];
    int* s_start = prep_smem;        // [E]
    int* s_end = s_start + E;        // [E]
    int* s_sb = s_end + E;           // [E + 1]: first global K-step of each expert, then the total
    __shared__ int s_flags;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    const int Mi = static_cast<int>(M);

    if (warp == 0) {
        int carry_end = 0, carry_steps = 0, flags = 0;
        for (int base = 0; base < E; base += 32) {
            const int g = base + lane;
            int o = 0;
            if (g < E) {
                o = offs[g];
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
    const int TS = s_sb[E];

    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            plan[0] = TS;
            plan[1] = E;
            if (s_flags) atomicOr(&g_device_status, s_flags);
        }
        int32_t* ex = plan + PLAN_HDR;
        int32_t* order = ex + 4 * E;
        for (int g = threadIdx.x; g < E; g += PREP_THREADS) {
            const int len = s_end[g] - s_start[g];
            ex[4 * g + 0] = s_start[g];
            ex[4 * g + 1] = len;
            ex[4 * g + 2] = (len + BK - 1) / BK;
            ex[4 * g + 3] = s_sb[g];
            int rank = 0;  // longest first; equal lengths keep expert order
            for (int h = 0; h < E; ++h) {
                const int lh = s_end[h] - s_start[h];
                rank += (lh > len) || (lh == len && h < g);
            }
            order[rank] = g;
        }
    }

    // Scale-factor gather as a tile transpose: a task is (128-row block rb,
    // 32 consecutive global K-steps). Lane l of a warp owns K-step gs0 + l and
    // loads that step's 4 scale bytes of one row, so consecutive lanes read
    // consecutive 4-byte groups of the row (coalesced within an expert); the
    // words are staged in a padded [128][33] shared tile, then each 512-byte
    // block is written by one warp with 16-byte stores.
    uint32_t* tile = reinterpret_cast<uint32_t*>(s_sb + E + 1);  // [PREP_ROWS][PREP_TILE_STEPS + 1]
    const int nchunks = (TS + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS;
    const long long ntasks = static_cast<long long>(ntn + 2 * ntk) * nchunks;
    const long long sM = M / 32;
    for (long long task = blockIdx.x; task < ntasks; task += gridDim.x) {
        const int rb = static_cast<int>(task / nchunks);
        const int gs0 = static_cast<int>(task - static_cast<long long>(rb) * nchunks) * PREP_TILE_STEPS;
        const uint8_t* plane;
        int rows, row0;
        uint8_t* dst;       // scale-factor block of global K-step 0 for this row block
        size_t dst_step;    // bytes between consecutive global K-steps
        if (rb < ntn) {
            plane = sA; rows = N; row0 = rb * BM;
            dst = sfa + static_cast<size_t>(rb) * ts_max * SF_ATOM;
            dst_step = SF_ATOM;
        } else {
            const int rbb = rb - ntn;
            plane = sB; rows = K; row0 = rbb * BM;
            dst = sfb + (static_cast<size_t>(rbb >> 1) * ts_max * 2 + (rbb & 1)) * SF_ATOM;
            dst_step = 2 * SF_ATOM;
        }
        // this lane's K-step: its expert, first scale column and valid 32-token blocks
        const int gs = gs0 + lane;
        long long col = 0;
        int nvalid = 0;
        if (gs < TS) {
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
        for (int r = warp; r < PREP_ROWS; r += PREP_THREADS / 32) {
            const int row = row0 + r;
            uint32_t wv = 0;
            if (row < rows) {
                const uint8_t* src = plane + static_cast<size_t>(row) * sM + col;
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
                    if (kb < nvalid) wv |= static_cast<uint32_t>(__ldg(src + kb)) << (8 * kb);
            }
            tile[r * (PREP_TILE_STEPS + 1) + lane] = wv;
        }
        __syncthreads();
        // block j of this task: lane r0 writes rows r0, r0+32, r0+64, r0+96 (16 bytes)
        for (int j = warp; j < PREP_TILE_STEPS; j += PREP_THREADS / 32) {
            if (gs0 + j >= TS) continue;
            uint4 o;
            o.x = tile[(lane + 0) * (PREP_TILE_STEPS + 1) + j];
            o.y = tile[(lane + 32) * (PREP_TILE_STEPS + 1) + j];
            o.z = tile[(lane + 64) * (PREP_TILE_STEPS + 1) + j];
            o.w = tile[(lane + 96) * (PREP_TILE_STEPS + 1) + j];
            reinterpret_cast<uint4*>(dst + static_cast<size_t>(gs0 + j) * dst_step)[lane] = o;
        }
        __syncthreads();
    }
    // This block's work is done: once every block got here the main kernel
    // may launch and run its prologue (it waits for this grid's completion
    // before reading anything written here). Triggering earlier would let its
    // resident CTAs crowd this kernel off the SMs.
    griddep_launch_dependents();
}

// ============================================================== main kernel

// One CTA pair (a 2-CTA cluster) owns a 256 x 256 output tile: rows
// [nt*256, nt*256+256) of A (the N axis) by rows [kt*256, kt*256+256) of B
// (the K axis). CTA r of the pair holds A rows nt*256 + 128r .. +128 and B
// rows kt*256 + 128r .. +128 in its shared memory, its own 128 accumulator
// rows in its TMEM, and stores those 128 output rows. The leader (r = 0)
// issues the M = 256 block-scaled MMAs for both; each SM then reads 32 KB of
// operands per K-step instead of the 48 KB a 128 x 256 single-CTA tile needs.
constexpr int PAIR_M = 2 * BM;    // 256 rows of A per pair tile
constexpr int HALF_N = BN / 2;    // 128 rows of B per CTA
constexpr int STAGES = 6;
constexpr int A_STAGE = BM * BK;       // 16 KB
constexpr int B_STAGE = HALF_N * BK;   // 16 KB
constexpr int SFA_STAGE = SF_ATOM;     // this CTA's 128 A rows
constexpr int SFB_STAGE = 2 * SF_ATOM; // all 256 B rows of the tile (each CTA's MMA half needs them)
constexpr uint32_t CTA_TX_BYTES = A_STAGE + B_STAGE + SFA_STAGE + SFB_STAGE;
constexpr uint32_t PAIR_TX_BYTES = 2 * CTA_TX_BYTES;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
constexpr int NUM_BARS = 2 * STAGES + 3;  // full[S], empty[S], tmem_full, tmem_empty, drain
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int MAIN_SMEM = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
constexpr int EPI_WARPS = 8;
constexpr int MAIN_THREADS = 32 * (3 + EPI_WARPS);  // producer, MMA issuer, stage watcher, epilogue
// Named barriers between the stage watcher and the MMA warp (64 threads each):
// BAR_READY + st: stage st holds data (watcher arrives, MMA warp syncs);
// BAR_FREE + st: the MMA warp has taken stage st (MMA warp arrives, watcher
// syncs before it signals that stage again), so arrivals and syncs on every
// id pair up one to one.
constexpr uint32_t BAR_READY = 1;
constexpr uint32_t BAR_FREE = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SFA = 256;  // + 4 * stage: 4 columns of A scales per stage
constexpr uint32_t TMEM_SFB = 288;  // + 8 * stage: 8 columns of B scales per stage

static_assert(OFF_B % 1024 == 0 && OFF_SFA % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(TMEM_SFA + 4 * STAGES <= TMEM_SFB && TMEM_SFB + 8 * STAGES <= TMEM_COLS, "TMEM budget");
static_assert(MAIN_SMEM <= 232448, "shared memory budget");
static_assert(BAR_READY + STAGES <= BAR_FREE && BAR_FREE + STAGES <= 16, "named barrier ids");

// Instruction descriptor, kind::mxf8f6f4: A and B E4M3 (0), both K-major,
// N >> 3 at bits 17-22, E8M0 scales (bit 23), M >> 4 at bits 24-28 (M = 256
// across the pair); the scale byte selectors for B (bits 4-5) and A (bits
// 29-30) are or-ed in per MMA.
constexpr uint32_t IDESC_BASE = (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                                (static_cast<uint32_t>(PAIR_M >> 4) << 24);

struct MainParams {
    const int32_t* plan;
    uint16_t* out;
    int E, N, K;
    int ts_max, ntn2, ntk;   // ntn2 = ceil(N / 256) pair-tile rows
    unsigned long long wait_ns;
    int stall_first_stage;   // test hook: over-declare the first stage's bytes so its wait runs out
};

// Bounded wait: returns false (and raises the CTA's abort flag and the device
// status word) if the phase does not complete within wait_ns, or returns
// false at once if another role of this CTA already aborted.
__device__ uint32_t g_suspend_ns = 0;  // try_wait suspend hint for waiting roles (0: plain polling)

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
    int g, nt, kt, start, len, nsteps, step_base;
};

// Work item i (in longest-expert-first order, the tiles of one expert
// consecutive, K-tiles fastest) -> expert and pair tile.
__device__ __forceinline__ Item load_item(const int32_t* __restrict__ plan, int E, int ntk, int nt_per_expert,
                                          long long i) {
    const int32_t* ex = plan + PLAN_HDR;
    const int32_t* order = ex + 4 * E;
    const int r = static_cast<int>(i / nt_per_expert);
    const int t = static_cast<int>(i - static_cast<long long>(r) * nt_per_expert);
    Item it;
    it.g = __ldg(order + r);
    it.nt = t / ntk;
    it.kt = t - it.nt * ntk;
    it.start = __ldg(ex + 4 * it.g + 0);
    it.len = __ldg(ex + 4 * it.g + 1);
    it.nsteps = __ldg(ex + 4 * it.g + 2);
    it.step_base = __ldg(ex + 4 * it.g + 3);
    return it;
}

// Next item of this pair's static schedule at or after pass `pass` (which is
// advanced past it), or -1 when the schedule is exhausted.
__device__ __forceinline__ long long item_index(long long pass, int G, int pair);
__device__ __forceinline__ long long next_item(long long& pass, int G, int pair, long long total) {
    while (pass * G < total) {
        const long long i = item_index(pass, G, pair);
        ++pass;
        if (i < total) return i;
    }
    return -1;
}

// Static schedule over CTA pairs: pass p hands items [p*G, (p+1)*G) to the
// pairs, reversing the direction on odd passes so that, with items sorted by
// cost, the loads even out (no atomics; a pair knows its items from its
// index alone, and both CTAs of a pair walk the same list).
__device__ __forceinline__ long long item_index(long long pass, int G, int pair) {
    return pass * G + ((pass & 1) ? (G - 1 - pair) : pair);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MAIN_THREADS, 1)
    wgrad_main(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
               const MainParams p) {
    extern __shared__ uint8_t main_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(main_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs), 1 = peer
    const bool leader = rank == 0;

    const uint32_t bar_full = sbase + OFF_BAR;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;
    const uint32_t bar_tempty = bar_tfull + 8;
    const uint32_t bar_drain = bar_tempty + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);    // leader's arrive.expect_tx for both CTAs' bytes
            mbar_init(bar_empty + 8 * s, 1);   // leader's MMA commit, multicast to both CTAs
        }
        mbar_init(bar_tfull, 1);               // leader's commit after a tile, multicast
        mbar_init(bar_tempty, 2 * EPI_WARPS);  // epilogue warps of both CTAs (leader's copy is used)
        mbar_init(bar_drain, 1);               // leader's final commit, multicast
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
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

    const int nt_per_expert = p.ntn2 * p.ntk;
    const long long total = static_cast<long long>(p.E) * nt_per_expert;
    const int G = gridDim.x / 2, pair = blockIdx.x / 2;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(bar_full, 0);
            uint32_t c = 0;
            bool ok = true;
            for (long long pass = 0; ok && pass * G < total; ++pass) {
                const long long i = item_index(pass, G, pair);
                if (i >= total) continue;
                const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
                const int a_row = it.nt * PAIR_M + static_cast<int>(rank) * BM;
                const int b_row = it.kt * BN + static_cast<int>(rank) * HALF_N;
                const int sfa_row = (it.nt * 2 + static_cast<int>(rank)) * p.ts_max + it.step_base;
                const int sfb_row = (it.kt * p.ts_max + it.step_base) * 2;
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const int st = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    // test hook: only the (over-declared) first fill is issued, so the
                    // stuck phase is never re-armed
                    if (p.stall_first_stage && c >= 1) { ok = false; break; }
                    if (!wait_phase(bar_empty + 8 * st, ph ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
                    const uint32_t fb = full_leader + 8 * st;
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * st, PAIR_TX_BYTES + (p.stall_first_stage ? 16u : 0u));
                    const int x = it.start + s * BK;
                    tma_load_2d_pair(sbase + OFF_A + st * A_STAGE, &tmA, fb, x, a_row);
                    tma_load_2d_pair(sbase + OFF_B + st * B_STAGE, &tmB, fb, x, b_row);
                    tma_load_2d_pair(sbase + OFF_SFA + st * SFA_STAGE, &tmSFA, fb, 0, sfa_row + s);
                    tma_load_2d_pair(sbase + OFF_SFB + st * SFB_STAGE, &tmSFB, fb, 0, sfb_row + 2 * s);
                }
            }
            if (leader && (!ok || *abort_flag)) {
                // let every copy still in flight land before the pair exits
                const uint32_t n = c < STAGES ? c : STAGES;
                for (uint32_t d = 1; d <= n; ++d) {
                    const uint32_t j = c - d;
                    drain_phase(bar_full + 8 * (j % STAGES), (j / STAGES) & 1, p.wait_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        // The whole warp walks the schedule; one elected lane issues each
        // tcgen05 operation. The per-stage loop reads no memory: a load or an
        // mbarrier probe here stalls this warp long enough to drain the
        // tensor pipe, so stage readiness arrives through named barriers from
        // the watcher warp. After an abort the loop still walks every stage
        // (skipping the tensor work) so that the named barriers stay paired.
        if (leader) {
            uint32_t c = 0, tiles = 0;
            bool live = true;
            // the next item's schedule entry is loaded one tile ahead, off the
            // tile-boundary critical path
            long long pass = 0;
            long long i_next = next_item(pass, G, pair, total);
            Item it_next = i_next >= 0 ? load_item(p.plan, p.E, p.ntk, nt_per_expert, i_next) : Item{};
            while (i_next >= 0) {
                const Item it = it_next;
                i_next = next_item(pass, G, pair, total);
                if (i_next >= 0) it_next = load_item(p.plan, p.E, p.ntk, nt_per_expert, i_next);
                if (it.nsteps == 0) continue;
                if (live) {
                    bool ok = true;
                    // both CTAs' epilogues have drained the accumulator; their arrivals
                    // only signal (the drained TMEM loads completed before them), so a
                    // CTA-scope acquire is enough
                    if (lane == 0) ok = !*abort_flag && wait_phase(bar_tempty, (tiles & 1) ^ 1, abort_flag, p.wait_ns);
                    live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
                tc_fence_after();
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const uint32_t st = c % STAGES;
                    named_bar_sync(BAR_READY + st, 64);
                    if (live) {
                        tc_fence_after();
                        const uint32_t sfa_t = tmem + TMEM_SFA + 4 * st;
                        const uint32_t sfb_t = tmem + TMEM_SFB + 8 * st;
                        const uint32_t sfa_s = sbase + OFF_SFA + st * SFA_STAGE;
                        const uint32_t sfb_s = sbase + OFF_SFB + st * SFB_STAGE;
                        tc_cp_32x128b_warpx4_pair_elect(sfa_t, desc_sf_block(sfa_s));
                        tc_cp_32x128b_warpx4_pair_elect(sfb_t, desc_sf_block(sfb_s));
                        tc_cp_32x128b_warpx4_pair_elect(sfb_t + 4, desc_sf_block(sfb_s + SF_ATOM));
                        const int rem = it.len - s * BK;
                        const int nk = rem >= BK ? 4 : (rem >> 5);
                        const uint32_t a_s = sbase + OFF_A + st * A_STAGE;
                        const uint32_t b_s = sbase + OFF_B + st * B_STAGE;
                        for (int kk = 0; kk < nk; ++kk) {
                            const uint32_t idesc = IDESC_BASE | (static_cast<uint32_t>(kk) << 29) |
                                                   (static_cast<uint32_t>(kk) << 4);
                            tc_mma_mxf8_pair_elect(tmem, desc_kmajor_sw128(a_s + 32 * kk),
                                                   desc_kmajor_sw128(b_s + 32 * kk), idesc, sfa_t, sfb_t,
                                                   (s > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit_pair_elect(bar_empty + 8 * st, 0x3);  // frees the stage in both CTAs
                    }
                    named_bar_arrive(BAR_FREE + st, 64);
                }
                if (live) {
                    tc_commit_pair_elect(bar_tfull, 0x3);  // both accumulator halves complete
                    ++tiles;
                }
            }
            // every MMA / copy issued for the pair has finished before teardown
            tc_commit_pair_elect(bar_drain, 0x3);
        }
        if (lane == 0) drain_phase(bar_drain, 0, p.wait_ns);
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ stage watcher (leader only)
        // Waits (bounded) for each stage's data and hands it to the MMA warp
        // through BAR_READY; after an abort it stops waiting but keeps the
        // barrier pairing until the schedule ends.
        if (leader) {
            uint32_t c = 0;
            bool live = true;
            for (long long pass = 0; pass * G < total; ++pass) {
                const long long i = item_index(pass, G, pair);
                if (i >= total) continue;
                const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const uint32_t st = c % STAGES;
                    if (c >= STAGES) named_bar_sync(BAR_FREE + st, 64);  // MMA warp took the previous fill
                    if (live) {
                        bool ok = true;
                        if (lane == 0) ok = wait_phase(bar_full + 8 * st, (c / STAGES) & 1, abort_flag, p.wait_ns);
                        live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    }
                    named_bar_arrive(BAR_READY + st, 64);
                }
            }
            // consume the MMA warp's last BAR_FREE arrivals so every id ends paired
            for (uint32_t d = c < STAGES ? c : STAGES; d > 0; --d) named_bar_sync(BAR_FREE + (c - d) % STAGES, 64);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (8 warps per CTA)
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = (warp - 3) >> 2;   // column half of the 256-wide tile
        const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
        uint32_t tiles = 0;
        for (long long pass = 0; pass * G < total; ++pass) {
            const long long i = item_index(pass, G, pair);
            if (i >= total) continue;
            const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
            const int row = it.nt * PAIR_M + static_cast<int>(rank) * BM + q * 32 + lane;
            const int col0 = it.kt * BN + h * 128;
            uint16_t* orow = p.out + (static_cast<size_t>(it.g) * p.N + row) * static_cast<size_t>(p.K) + col0;
            if (it.nsteps == 0) {
                // expert without tokens: exact +0.0 slab
                if (row < p.N) {
                    for (int c = 0; c < 128; c += 8)
                        if (col0 + c < p.K) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            // one lane waits, the warp follows its verdict (the TMEM loads below
            // are warp-collective, so the lanes must not split on a timeout)
            bool ready = true;
            if (lane == 0) ready = wait_phase(bar_tfull, tiles & 1, abort_flag, p.wait_ns);
            if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) break;
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(taddr + 32 * j, v[j]);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 4; ++j) reg_fence(v[j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // this CTA's accumulator half may be overwritten
                if (leader) mbar_arrive(bar_tempty);
                else mbar_arrive_cluster(tempty_leader);
            }
            ++tiles;
            if (row < p.N) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        if (col0 + 32 * j + c < p.K) {
                            uint4 o;
                            o.x = pack_bf16x2(v[j][c + 0], v[j][c + 1]);
                            o.y = pack_bf16x2(v[j][c + 2], v[j][c + 3]);
                            o.z = pack_bf16x2(v[j][c + 4], v[j][c + 5]);
                            o.w = pack_bf16x2(v[j][c + 6], v[j][c + 7]);
                            *reinterpret_cast<uint4*>(orow + 32 * j + c) = o;
                        }
                    }
                }
            }
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

bool ws_layout(int E, int N, int K, int64_t M, WsLayout* L) {
    if (E < 1 || E > MXFP8_MAX_EXPERTS || N < 1 || K < 1 || M < 32 || (M % 32) != 0) return false;
    if (M > (int64_t(1) << 31) - 256) return false;
    L->ntn = (N + BM - 1) / BM;
    L->ntk = (K + BN - 1) / BN;
    const int64_t ts = (M + BK - 1) / BK + E;
    if (ts > (int64_t(1) << 30)) return false;
    L->ts_max = static_cast<int>(ts);
    const size_t plan_bytes = sizeof(int32_t) * (PLAN_HDR + 5 * static_cast<size_t>(E));
    L->plan_off = 0;
    L->sfa_off = (plan_bytes + 1023) & ~size_t(1023);
    L->sfb_off = L->sfa_off + static_cast<size_t>(L->ntn) * L->ts_max * SF_ATOM;
    L->total = L->sfb_off + static_cast<size_t>(L->ntk) * L->ts_max * 2 * SF_ATOM;
    return true;
}

cudaError_t launch_wgrad(const WgradArgs& a, const CUtensorMap* maps, const char** what) {
    const WsLayout& L = a.lay;
    int32_t* plan = reinterpret_cast<int32_t*>(a.ws + L.plan_off);
    uint8_t* sfa = a.ws + L.sfa_off;
    uint8_t* sfb = a.ws + L.sfb_off;

    *what = "plan / scale re-layout kernel";
    {
        // enough blocks for every task of the largest possible plan, at most 4 per SM
        const long long tasks = static_cast<long long>(L.ntn + 2 * L.ntk) *
                                ((L.ts_max + PREP_TILE_STEPS - 1) / PREP_TILE_STEPS);
        long long blocks = tasks;
        if (blocks > 4LL * a.num_sms) blocks = 4LL * a.num_sms;
        if (blocks < 1) blocks = 1;
        const size_t sm = sizeof(int) * (3 * static_cast<size_t>(a.E) + 1) +
                          sizeof(uint32_t) * PREP_ROWS * (PREP_TILE_STEPS + 1);
        wgrad_prep<<<static_cast<unsigned>(blocks), PREP_THREADS, sm, a.stream>>>(
            a.offs, a.sA, a.sB, plan, sfa, sfb, a.E, a.N, a.K, a.M, L.ts_max, L.ntn, L.ntk);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    *what = "main contraction kernel";
    // per device: the shared-memory opt-in and the number of CTA pairs that
    // can be resident at once (the persistent grid)
    static int max_pairs[64] = {};
    if (a.dev < 0 || a.dev >= 64) return cudaErrorInvalidDevice;
    if (max_pairs[a.dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(wgrad_main, cudaFuncAttributeMaxDynamicSharedMemorySize, MAIN_SMEM);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * (a.num_sms / 2));
        q.blockDim = dim3(MAIN_THREADS);
        q.dynamicSmemBytes = MAIN_SMEM;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, wgrad_main, &q);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        max_pairs[a.dev] = clusters;
    }
    MainParams mp;
    mp.plan = plan;
    mp.out = a.out;
    mp.E = a.E;
    mp.N = a.N;
    mp.K = a.K;
    mp.ts_max = L.ts_max;
    mp.ntn2 = (a.N + PAIR_M - 1) / PAIR_M;
    mp.ntk = L.ntk;
    mp.wait_ns = a.wait_limit_ns;
    mp.stall_first_stage = a.stall_first_stage;
    const long long total = static_cast<long long>(a.E) * mp.ntn2 * mp.ntk;
    const int pairs = static_cast<int>(total < max_pairs[a.dev] ? total : max_pairs[a.dev]);
    if (a.ev_before) {
        cudaError_t e = cudaEventRecord(a.ev_before, a.stream);
        if (e != cudaSuccess) return e;
    }
    // programmatic dependent launch: the prologue (barriers, TMEM allocation,
    // descriptor prefetch) overlaps the prep kernel; griddepcontrol.wait in
    // the kernel orders every read of the prep kernel's output after it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(MAIN_THREADS);
    cfg.dynamicSmemBytes = MAIN_SMEM;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, wgrad_main, maps[0], maps[1], maps[2], maps[3], mp);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ev_after) {
        e = cudaEventRecord(a.ev_after, a.stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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
