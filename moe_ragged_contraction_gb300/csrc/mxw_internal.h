// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxw {

// A CTA pair owns a 256 x TN output tile (TN <= MAX_TN); the token axis is
// walked in K-steps of BK tokens ("Ragged MXFP8 Weight Gradients", section 1:
// a pipelined kernel walks the contraction in fixed steps of 128 tokens along
// M). BM is the share of one CTA of the pair's 256 "M-side" rows.
constexpr int BM = 128;
constexpr int MAX_TN = 448;
constexpr int BK = 128;
constexpr int SF_ATOM = 512;  // bytes of scale factors for 128 rows x one K-step

// Schedule ("plan") layout in the workspace, int32 words:
//   [0] total K-steps over all experts, [1] E,
//   [PLAN_HDR + 4g + {0,1,2,3}] = start, length, K-steps, first global K-step of expert g,
//   [PLAN_HDR + 4E + r]        = expert with the r-th longest token run.
constexpr int PLAN_HDR = 8;

// Tile orientation and sizes. kn == 0: the pair's 256-row "M side" runs over
// the rows of A (output rows n) and the TN-row "N side" over the rows of B
// (output columns k); kn == 1 swaps them (the accumulator then holds the tile
// transposed). tn = n1 + n2: the widths of the one or two MMAs per 32-token
// chunk (n1 = min(tn, 256)); nblk_n = ceil(tn / 128) scale blocks per N-side
// tile; tiles_m = ceil(rows of the M side / 256), tiles_n = ceil(rows of the
// N side / tn).
// m_fastest: the order of one expert's tiles in the schedule (weight
// gradient). A pass of the persistent grid covers a run of consecutive tiles,
// so the operand indexed by the faster-moving tile index is read in full by
// every pass over the expert while the other is read about once: the faster
// index runs over the side with fewer rows (1: the M side, else the N side).
struct TileConfig {
    int kn, tn, n1, n2, nblk_n, tiles_m, tiles_n;
    int m_fastest;
};

// force: 0 = the orientation the kernel's cost model prefers (ties: kn == 0),
// 1 = kn == 0, 2 = kn == 1. force_tn: 0 = the modelled best tn of that
// orientation, else that tn (a multiple of 16 in [16, MAX_TN]). E and M (the
// mean run length) weigh the per-tile overhead. Returns false for invalid
// sizes or an invalid force_tn.
bool choose_tiles(int N, int K, int E, int64_t M, int force, int force_tn, TileConfig* tc);

// Workspace: the plan, then the M side's scale-factor blocks
// [tiles_m][ts_max][2][512 B], then the N side's [tiles_n][ts_max][nblk_n][512 B].
struct WsLayout {
    size_t plan_off, sfm_off, sfn_off, total;
    int ts_max;  // upper bound on the total number of K-steps
    TileConfig tc;
};

// Workspace layout for these sizes and tiles; returns false if unsupported.
bool ws_layout(int E, int N, int K, int64_t M, const TileConfig& tc, WsLayout* out);

// Largest workspace over both orientations (0 if the sizes are invalid).
size_t ws_bytes_any_orientation(int E, int N, int K, int64_t M, int force_tn);

struct WgradArgs {
    const uint8_t *A, *sA, *B, *sB;
    const int32_t* offs;
    int E, N, K;
    int64_t M;
    uint16_t* out;
    uint8_t* ws;
    WsLayout lay;
    int dev, num_sms;
    uint64_t wait_limit_ns;
    cudaStream_t stream;
    cudaEvent_t ev_before, ev_after;
    int stall_first_stage;  // failure-path test hook (0 in normal use)
    int tma_store;          // maps[5] describes out: TMA-store epilogue where its staging fits
    int grid;               // 1: K-steps on the global 128-token grid (scale blocks per grid step)
    int gather;             // 1: the prep kernel lays the scale planes out into the workspace;
                            // 0: maps[3], maps[4] describe the caller's blocks (grid == 1,
                            // lay.ts_max = grid steps) and the prep writes the plan only
};

// Enqueue the plan / scale re-layout kernel and the main contraction kernel.
// maps: the M-side operand (boxes of BM rows x BK tokens), the N-side operand
// for the first and the second MMA (n1/2 and n2/2 rows x BK tokens; the second
// is unused when n2 == 0), all with the 128-byte swizzle, and the two sides'
// scale-factor blocks viewed as u32 [blocks][128] (boxes of 1 and nblk_n
// blocks). Returns a cudaError_t; `what` names the step.
cudaError_t launch_wgrad(const WgradArgs& a, const CUtensorMap* maps, const char** what);

// Grouped GEMM (non-contracting ragged dot): out[t][n] = sum_k x(t,k) w(g,n,k)
// for the rows t of group g; X [M][K], W [E][N][K] E4M3 with scales along k.
// Tiles: 256 rows of X (a row tile never crosses a group) by tn rows of W[g].
// Workspace: the plan (row-tile table), then the row tiles' scale-factor
// blocks [mtiles_max][ksteps][2][512 B], then the weights' [E * tiles_n][ksteps][nblk_n][512 B].
struct GemmLayout {
    size_t plan_off, sfm_off, sfn_off, total;
    int mtiles_max, ksteps;  // row tiles over every routing: ceil(M / 256) + E
    TileConfig tc;
};

bool choose_gemm_tiles(int N, int K, int E, int64_t M, int force_tn, TileConfig* tc);
bool gemm_layout(int E, int N, int K, int64_t M, const TileConfig& tc, GemmLayout* out);

struct GemmArgs {
    const uint8_t *X, *sX, *W, *sW;
    const int32_t* offs;
    int E, N, K;
    int64_t M;
    uint16_t* out;
    uint8_t* ws;
    GemmLayout lay;
    int dev, num_sms;
    uint64_t wait_limit_ns;
    cudaStream_t stream;
    cudaEvent_t ev_before, ev_after;
    int tma_store;          // as in WgradArgs
};

// maps: X (boxes of BM rows x BK), W as 3-D [E][N][K] (boxes of n1/2 and n2/2
// rows), and the scale-factor blocks as u32 [blocks][128] (boxes of 1 and nblk_n).
cudaError_t launch_gemm(const GemmArgs& a, const CUtensorMap* maps, const char** what);

cudaError_t launch_quantize(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, cudaStream_t stream);
cudaError_t launch_quantize_transpose(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s,
                                      cudaStream_t stream);
// As launch_quantize_transpose, writing the scales also (or only: s may be
// null) as tcgen05 scale-factor blocks for tiles of tile_rows rows on the
// global 128-token grid (sf: [ceil(R / tile_rows)][ceil(M / 128)][ceil(tile_rows / 128)][512 B]).
cudaError_t launch_quantize_transpose_sf(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s, uint8_t* sf,
                                         int tile_rows, cudaStream_t stream);

// Loads the module holding the weight-gradient kernels on the current device
// (the runtime otherwise loads it at the first launch), without launching.
cudaError_t load_kernel_modules();

// Sets the calling thread's mxfp8_last_error() message; returns `code`.
int set_last_error(int code, const char* msg);

// Suspend hint (ns) for the kernels' mbarrier waits on the current device.
cudaError_t set_suspend_hint(uint32_t ns);

// Device status word (MXFP8_DEV_* bits).
cudaError_t read_device_status(int32_t* status, int clear);

}  // namespace mxw
