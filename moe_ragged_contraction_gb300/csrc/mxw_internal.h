// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxw {

// Output tile of one CTA: BM rows of A (the N axis) x BN rows of B (the K
// axis); the token axis is walked in K-steps of BK tokens ("Ragged MXFP8
// Weight Gradients", section 1: a pipelined kernel walks the contraction in
// fixed steps of 128 tokens along M).
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int SF_ATOM = 512;  // bytes of scale factors for 128 rows x one K-step

// Schedule ("plan") layout in the workspace, int32 words:
//   [0] total K-steps over all experts, [1] E,
//   [PLAN_HDR + 4g + {0,1,2,3}] = start, length, K-steps, first global K-step of expert g,
//   [PLAN_HDR + 4E + r]        = expert with the r-th longest token run.
constexpr int PLAN_HDR = 8;

struct WsLayout {
    size_t plan_off, sfa_off, sfb_off, total;
    int ts_max;  // upper bound on the total number of K-steps
    int ntn, ntk;
};

// Workspace layout for these sizes; returns false if the sizes are invalid.
bool ws_layout(int E, int N, int K, int64_t M, WsLayout* out);

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
};

// Rows of A and of B that one CTA loads per K-step (the CTA's half of a
// 256 x 256 pair tile).
constexpr int HALF_TILE_ROWS = 128;

// Enqueue the plan / scale re-layout kernel and the main contraction kernel.
// maps: A and B operand tiles (HALF_TILE_ROWS rows x BK tokens, 128-byte
// swizzle) and the scale-factor workspaces viewed as u32 [blocks][128]
// (boxes of 1 and 2 blocks). Returns a cudaError_t; `what` names the step.
cudaError_t launch_wgrad(const WgradArgs& a, const CUtensorMap* maps, const char** what);

cudaError_t launch_quantize(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, cudaStream_t stream);

// Sets the calling thread's mxfp8_last_error() message; returns `code`.
int set_last_error(int code, const char* msg);

// Suspend hint (ns) for the kernels' mbarrier waits on the current device.
cudaError_t set_suspend_hint(uint32_t ns);

// Device status word (MXFP8_DEV_* bits).
cudaError_t read_device_status(int32_t* status, int clear);

}  // namespace mxw
