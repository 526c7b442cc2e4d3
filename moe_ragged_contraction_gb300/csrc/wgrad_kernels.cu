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
constexpr int PREP_WARPS = PREP_THREADS / 32;

// grid: x = ceil(ts_max / PREP_WARPS) groups of K-steps, y = ntn + 2 * ntk
// 128-row blocks (A blocks first, then B blocks). Each warp writes one
// 512-byte scale-factor block: lane r0 writes bytes [16 r0, 16 r0 + 16),
// holding rows r0 + 32 j (j = 0..3) x 4 consecutive 32-token blocks.
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

    if (blockIdx.x == 0 && blockIdx.y == 0) {
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

    const int gs = blockIdx.x * PREP_WARPS + warp;  // global K-step of this warp
    if (gs >= TS) return;
    // expert owning global K-step gs: the last g with s_sb[g] <= gs
    int lo = 0, hi = E;  // invariant: s_sb[lo] <= gs < s_sb[hi] (s_sb[E] = TS)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_sb[mid] <= gs) lo = mid; else hi = mid;
    }
    const int g = lo;
    const long long t0 = static_cast<long long>(s_start[g]) + static_cast<long long>(gs - s_sb[g]) * BK;
    const long long tend = s_end[g];

    const int rb = blockIdx.y;
    const uint8_t* plane;
    int rows, row0;
    uint8_t* dst;
    if (rb < ntn) {
        plane = sA; rows = N; row0 = rb * BM;
        dst = sfa + (static_cast<size_t>(rb) * ts_max + gs) * SF_ATOM;
    } else {
        const int rbb = rb - ntn;
        plane = sB; rows = K; row0 = rbb * BM;
        dst = sfb + ((static_cast<size_t>(rbb >> 1) * ts_max + gs) * 2 + (rbb & 1)) * SF_ATOM;
    }
    const long long sM = M / 32;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int row = row0 + lane + 32 * j;
        uint32_t word = 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            const long long t = t0 + 32 * kb;
            if (row < rows && t < tend) {
                const uint32_t b = __ldg(plane + static_cast<size_t>(row) * sM + (t >> 5));
                word |= b << (8 * kb);
            }
        }
        w[j] = word;
    }
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
}

// ============================================================== main kernel

constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK;   // 16 KB
constexpr int B_STAGE = BN * BK;   // 32 KB
constexpr int SFA_STAGE = SF_ATOM;
constexpr int SFB_STAGE = 2 * SF_ATOM;
constexpr uint32_t TX_BYTES = A_STAGE + B_STAGE + SFA_STAGE + SFB_STAGE;
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
constexpr int MAIN_THREADS = 32 * (2 + EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SFA = 256;  // + 4 * stage: 4 columns of A scales per stage
constexpr uint32_t TMEM_SFB = 288;  // + 8 * stage: 8 columns of B scales per stage

static_assert(OFF_B % 1024 == 0 && OFF_SFA % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(TMEM_SFB + 8 * STAGES <= TMEM_COLS, "TMEM budget");

// Instruction descriptor, kind::mxf8f6f4: A and B E4M3 (0), both K-major,
// N >> 3 at bits 17-22, E8M0 scales (bit 23), M >> 4 at bits 24-28; the scale
// byte selectors for B (bits 4-5) and A (bits 29-30) are or-ed in per MMA.
constexpr uint32_t IDESC_BASE = (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                                (static_cast<uint32_t>(BM >> 4) << 24);

struct MainParams {
    const int32_t* plan;
    const uint8_t* sfa;
    const uint8_t* sfb;
    uint16_t* out;
    int E, N, K;
    int ts_max, ntn, ntk;
    unsigned long long wait_ns;
};

// Bounded wait: returns false (and raises the CTA's abort flag and the device
// status word) if the phase does not complete within wait_ns, or returns
// false at once if another role already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned long long wait_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > wait_ns) {
            *abort_flag = 1;
            atomicOr(&g_device_status, MXFP8_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait used while tearing down after an abort (ignores the flag).
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

// Work item i (in longest-expert-first order, tiles of one expert
// consecutive, K-tiles fastest) -> expert and tile.
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

// Static schedule: pass p hands items [p*G, (p+1)*G) to the CTAs, reversing
// the direction on odd passes so that, with items sorted by cost, the loads
// even out (no atomics; every CTA knows its items from its index alone).
__device__ __forceinline__ long long item_index(long long pass, int G, int cta) {
    return pass * G + ((pass & 1) ? (G - 1 - cta) : cta);
}

__global__ void __launch_bounds__(MAIN_THREADS, 1)
    wgrad_main(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const MainParams p) {
    extern __shared__ uint8_t main_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(main_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar_full = sbase + OFF_BAR;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;
    const uint32_t bar_tempty = bar_tfull + 8;
    const uint32_t bar_drain = bar_tempty + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_tempty, EPI_WARPS);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nt_per_expert = p.ntn * p.ntk;
    const long long total = static_cast<long long>(p.E) * nt_per_expert;
    const int G = gridDim.x, cta = blockIdx.x;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t c = 0;
            bool ok = true;
            for (long long pass = 0; ok && pass * G < total; ++pass) {
                const long long i = item_index(pass, G, cta);
                if (i >= total) continue;
                const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const int st = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    if (!wait_phase(bar_empty + 8 * st, ph ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
                    const uint32_t fb = bar_full + 8 * st;
                    mbar_arrive_expect_tx(fb, TX_BYTES);
                    const int x = it.start + s * BK;
                    tma_load_2d(sbase + OFF_A + st * A_STAGE, &tmA, fb, x, it.nt * BM);
                    tma_load_2d(sbase + OFF_B + st * B_STAGE, &tmB, fb, x, it.kt * BN);
                    const size_t gstep = static_cast<size_t>(it.step_base + s);
                    bulk_g2s(sbase + OFF_SFA + st * SFA_STAGE,
                             p.sfa + (static_cast<size_t>(it.nt) * p.ts_max + gstep) * SF_ATOM, SFA_STAGE, fb);
                    bulk_g2s(sbase + OFF_SFB + st * SFB_STAGE,
                             p.sfb + (static_cast<size_t>(it.kt) * p.ts_max + gstep) * (2 * SF_ATOM), SFB_STAGE, fb);
                }
            }
            if (!ok || *abort_flag) {
                // let every copy still in flight land before the CTA exits
                const uint32_t n = c < STAGES ? c : STAGES;
                for (uint32_t d = 1; d <= n; ++d) {
                    const uint32_t j = c - d;
                    drain_phase(bar_full + 8 * (j % STAGES), (j / STAGES) & 1, p.wait_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t c = 0, tiles = 0;
            bool ok = true;
            for (long long pass = 0; ok && pass * G < total; ++pass) {
                const long long i = item_index(pass, G, cta);
                if (i >= total) continue;
                const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
                if (it.nsteps == 0) continue;
                if (!wait_phase(bar_tempty, (tiles & 1) ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                for (int s = 0; s < it.nsteps; ++s, ++c) {
                    const int st = c % STAGES;
                    const uint32_t ph = (c / STAGES) & 1;
                    if (!wait_phase(bar_full + 8 * st, ph, abort_flag, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + TMEM_SFA + 4 * st;
                    const uint32_t sfb_t = tmem + TMEM_SFB + 8 * st;
                    const uint32_t sfa_s = sbase + OFF_SFA + st * SFA_STAGE;
                    const uint32_t sfb_s = sbase + OFF_SFB + st * SFB_STAGE;
                    tc_cp_32x128b_warpx4(sfa_t, desc_sf_block(sfa_s));
                    tc_cp_32x128b_warpx4(sfb_t, desc_sf_block(sfb_s));
                    tc_cp_32x128b_warpx4(sfb_t + 4, desc_sf_block(sfb_s + SF_ATOM));
                    const int rem = it.len - s * BK;
                    const int nk = rem >= BK ? 4 : (rem >> 5);
                    const uint32_t a_s = sbase + OFF_A + st * A_STAGE;
                    const uint32_t b_s = sbase + OFF_B + st * B_STAGE;
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint32_t idesc = IDESC_BASE | (static_cast<uint32_t>(kk) << 29) |
                                               (static_cast<uint32_t>(kk) << 4);
                        tc_mma_mxf8(tmem, desc_kmajor_sw128(a_s + 32 * kk), desc_kmajor_sw128(b_s + 32 * kk), idesc,
                                    sfa_t, sfb_t, (s > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar_empty + 8 * st);  // frees the stage once these MMAs have read it
                }
                if (!ok) break;
                tc_commit(bar_tfull);  // accumulator complete
                ++tiles;
            }
            // every MMA / copy this thread issued has finished before teardown
            tc_commit(bar_drain);
            drain_phase(bar_drain, 0, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (8 warps)
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;   // column half of the 256-wide tile
        uint32_t tiles = 0;
        for (long long pass = 0; pass * G < total; ++pass) {
            const long long i = item_index(pass, G, cta);
            if (i >= total) continue;
            const Item it = load_item(p.plan, p.E, p.ntk, nt_per_expert, i);
            const int row = it.nt * BM + q * 32 + lane;
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
            if (!wait_phase(bar_tfull, tiles & 1, abort_flag, p.wait_ns)) break;
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
            if (lane == 0) mbar_arrive(bar_tempty);  // accumulator may be overwritten
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

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
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

cudaError_t launch_wgrad(const WgradArgs& a, const CUtensorMap& mapA, const CUtensorMap& mapB, const char** what) {
    const WsLayout& L = a.lay;
    int32_t* plan = reinterpret_cast<int32_t*>(a.ws + L.plan_off);
    uint8_t* sfa = a.ws + L.sfa_off;
    uint8_t* sfb = a.ws + L.sfb_off;

    *what = "plan / scale re-layout kernel";
    {
        dim3 grid((L.ts_max + PREP_WARPS - 1) / PREP_WARPS, L.ntn + 2 * L.ntk);
        const size_t sm = sizeof(int) * (3 * static_cast<size_t>(a.E) + 1);
        wgrad_prep<<<grid, PREP_THREADS, sm, a.stream>>>(a.offs, a.sA, a.sB, plan, sfa, sfb, a.E, a.N, a.K, a.M,
                                                         L.ts_max, L.ntn, L.ntk);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    *what = "main contraction kernel";
    static bool attr_set[64] = {};  // the attribute is set once per device
    if (a.dev < 0 || a.dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[a.dev]) {
        cudaError_t e = cudaFuncSetAttribute(wgrad_main, cudaFuncAttributeMaxDynamicSharedMemorySize, MAIN_SMEM);
        if (e != cudaSuccess) return e;
        attr_set[a.dev] = true;
    }
    MainParams mp;
    mp.plan = plan;
    mp.sfa = sfa;
    mp.sfb = sfb;
    mp.out = a.out;
    mp.E = a.E;
    mp.N = a.N;
    mp.K = a.K;
    mp.ts_max = L.ts_max;
    mp.ntn = L.ntn;
    mp.ntk = L.ntk;
    mp.wait_ns = a.wait_limit_ns;
    const long long total = static_cast<long long>(a.E) * L.ntn * L.ntk;
    const int grid = static_cast<int>(total < a.num_sms ? total : a.num_sms);
    if (a.ev_before) {
        cudaError_t e = cudaEventRecord(a.ev_before, a.stream);
        if (e != cudaSuccess) return e;
    }
    wgrad_main<<<grid, MAIN_THREADS, MAIN_SMEM, a.stream>>>(mapA, mapB, mp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ev_after) {
        e = cudaEventRecord(a.ev_after, a.stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

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
