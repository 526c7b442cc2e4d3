// C ABI of the library: argument validation, tensor-map creation, the
// per-(device, stream) scratch cache, and status / error reporting.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "mxw_internal.h"
#include "../../include/mxfp8_wgrad.h"

// 1: the regular entry points also run each expert's K-steps on the global
// 128-token grid: the prep's scale gather then does not depend on the routing
// (it starts at the kernel's entry, only the plan waits for offs) and the
// operand tiles start on 128-byte boundaries. Measured on GB300 against
// K-steps that start at each run's first token (same output bits),
// back-to-back throughput in one call: 671B down +1.4%, 671B up/gate +2.4%,
// 16B +1.9%, 16B production +2.2%.
#ifndef MXW_GRID_KSTEPS
#define MXW_GRID_KSTEPS 1
#endif

namespace {

thread_local char g_err[512] = "no error";
thread_local cudaEvent_t g_ev_before = nullptr;
thread_local cudaEvent_t g_ev_after = nullptr;
thread_local int g_stall_next = 0;

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int fail_cuda(cudaError_t e, const char* what) {
    return fail(MXFP8_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
    bool valid = false;
    int major = 0, minor = 0, sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Device checks: an sm_103 (GB300) GPU, the only target the library is built for.
int current_device(int* dev, DeviceInfo* info) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= 64) return fail(MXFP8_EUNSUPPORTED, "device index %d out of range", *dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[*dev];
    if (!d.valid) {
        e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, *dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, *dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
        d.valid = true;
    }
    *info = d;
    if (d.major != 10 || d.minor != 3)
        return fail(MXFP8_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", *dev,
                    d.major, d.minor);
    return MXFP8_OK;
}

int get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            return fail(MXFP8_ECUDA, "cuTensorMapEncodeTiled entry point unavailable (%s)", cudaGetErrorString(e));
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return MXFP8_OK;
}

// Token-contiguous E4M3 operand [rows][M] -> box of box_rows rows x 128 tokens,
// 128-byte swizzle; out-of-range rows and tokens read as zero.
int make_operand_map(CUtensorMap* map, const uint8_t* base, int rows, int64_t M, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = get_encoder(&enc);
    if (rc) return rc;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(M)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(mxw::BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MXFP8_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return MXFP8_OK;
}

// E4M3 operand [depth][rows][row_len] (row_len contiguous) -> 3-D boxes of
// box_rows rows x 128 elements x 1, 128-byte swizzle; out-of-range rows and
// columns read as zero (rows past `rows` never reach the next depth slice).
int make_operand_map3(CUtensorMap* map, const uint8_t* base, int64_t row_len, int rows, int depth, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = get_encoder(&enc);
    if (rc) return rc;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_len), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_len), static_cast<cuuint64_t>(row_len) * rows};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(mxw::BK), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MXFP8_ECUDA, "cuTensorMapEncodeTiled (3-D) failed (CUresult %d)", static_cast<int>(r));
    return MXFP8_OK;
}

// bf16 output viewed as [depth][rows][cols] for the TMA-store epilogue: boxes
// of 32 columns x 32 rows x 1, 64-byte swizzle (the staging layout the
// epilogue writes). Returns 0 when the layout does not allow a tensor map
// (rows of cols bf16 not a multiple of 16 bytes, or out not 16-byte aligned).
int make_out_map(CUtensorMap* map, uint16_t* out, int64_t cols, int64_t rows, int64_t depth) {
    if ((cols % 8) != 0 || (reinterpret_cast<uintptr_t>(out) & 15u) != 0) return 0;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (get_encoder(&enc)) return 0;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(cols) * rows * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 1 : 0;
}

// Scale-factor workspace viewed as u32 [blocks][128] (one 512-byte block per
// row); boxes of box_blocks whole blocks, no swizzle.
int make_sf_map(CUtensorMap* map, const uint8_t* base, int64_t blocks, int box_blocks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = get_encoder(&enc);
    if (rc) return rc;
    cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(blocks)};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_blocks)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MXFP8_ECUDA, "cuTensorMapEncodeTiled (scales) failed (CUresult %d)", static_cast<int>(r));
    return MXFP8_OK;
}

// Scratch cache keyed by (device, stream). Growth frees the old block in
// stream order and allocates the new one in stream order, so earlier calls
// on the same stream finish with the old block first. While the stream is
// being captured into a CUDA graph the cache neither grows nor frees (a
// captured allocation would belong to the graph, and the cache would keep a
// pointer the graph owns): a call that needs more scratch than the stream's
// cached block fails with MXFP8_ENOWS before anything is recorded.
struct WsEntry {
    int dev;
    cudaStream_t stream;
    void* ptr;
    size_t bytes;
};
std::vector<WsEntry> g_ws;

int cached_workspace(int dev, cudaStream_t stream, size_t need, void** out) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ec = cudaStreamIsCapturing(stream, &cap);
    if (ec != cudaSuccess) return fail_cuda(ec, "cudaStreamIsCapturing");
    std::lock_guard<std::mutex> lk(g_mu);
    for (WsEntry& w : g_ws) {
        if (w.dev == dev && w.stream == stream) {
            if (w.bytes >= need) {
                *out = w.ptr;
                return MXFP8_OK;
            }
            break;
        }
    }
    if (cap != cudaStreamCaptureStatusNone)
        return fail(MXFP8_ENOWS,
                    "the stream is being captured and the scratch cached for it holds less than the %zu bytes this "
                    "call needs: pass a workspace (the _ws entry point) or make the same call once on this stream "
                    "before capturing",
                    need);
    for (WsEntry& w : g_ws) {
        if (w.dev == dev && w.stream == stream) {
            cudaError_t e = cudaFreeAsync(w.ptr, stream);
            if (e != cudaSuccess) return fail_cuda(e, "cudaFreeAsync (workspace)");
            w.ptr = nullptr;
            w.bytes = 0;
            e = cudaMallocAsync(&w.ptr, need, stream);
            if (e != cudaSuccess) return fail_cuda(e, "cudaMallocAsync (workspace)");
            w.bytes = need;
            *out = w.ptr;
            return MXFP8_OK;
        }
    }
    WsEntry w{dev, stream, nullptr, 0};
    cudaError_t e = cudaMallocAsync(&w.ptr, need, stream);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMallocAsync (workspace)");
    w.bytes = need;
    g_ws.push_back(w);
    *out = w.ptr;
    return MXFP8_OK;
}

// Tile orientation mode (mxfp8_wgrad_set_tile_orientation); the initial value
// comes from MXFP8_TILE_ORIENTATION ("auto", "nk" or "kn"; default auto).
std::atomic<int> g_orientation{-1};
// N-side tile rows forced by mxfp8_wgrad_set_tile_rows (0 = modelled best);
// the initial value comes from MXFP8_TILE_ROWS (ignored unless admissible).
std::atomic<int> g_tile_rows{-1};
// Epilogue stores (mxfp8_wgrad_set_epilogue_store): 0 = TMA stores where their
// staging fits, 1 = direct stores only; the initial value comes from
// MXFP8_EPILOGUE_STORE ("auto" or "direct"; default auto).
std::atomic<int> g_store_mode{-1};

int store_mode() {
    int m = g_store_mode.load(std::memory_order_relaxed);
    if (m < 0) {
        const char* s = getenv("MXFP8_EPILOGUE_STORE");
        int v = (s && strcmp(s, "direct") == 0) ? 1 : 0;
        int expected = -1;
        g_store_mode.compare_exchange_strong(expected, v);
        m = g_store_mode.load(std::memory_order_relaxed);
    }
    return m;
}

int orientation_mode() {
    int m = g_orientation.load(std::memory_order_relaxed);
    if (m < 0) {
        const char* s = getenv("MXFP8_TILE_ORIENTATION");
        int v = 0;
        if (s && (s[0] == 'n' || s[0] == 'N')) v = 1;
        if (s && (s[0] == 'k' || s[0] == 'K')) v = 2;
        int expected = -1;
        g_orientation.compare_exchange_strong(expected, v);
        m = g_orientation.load(std::memory_order_relaxed);
    }
    return m;
}

int tile_rows_setting() {
    int t = g_tile_rows.load(std::memory_order_relaxed);
    if (t < 0) {
        const char* s = getenv("MXFP8_TILE_ROWS");
        int v = s ? atoi(s) : 0;
        if (v < 16 || v > mxw::MAX_TN || v % 16 != 0) v = 0;
        int expected = -1;
        g_tile_rows.compare_exchange_strong(expected, v);
        t = g_tile_rows.load(std::memory_order_relaxed);
    }
    return t;
}

uint64_t wait_limit_ns() {
    static uint64_t v = [] {
        const char* s = getenv("MXFP8_WAIT_LIMIT_MS");
        long long ms = s ? atoll(s) : 1000;
        if (ms < 1) ms = 1;
        if (ms > 60000) ms = 60000;
        return static_cast<uint64_t>(ms) * 1000000ull;
    }();
    return v;
}

int validate(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const int32_t* offs, int E,
             int N, int K, int64_t M, const uint16_t* out) {
    if (E < 0 || E > MXFP8_MAX_EXPERTS) return fail(MXFP8_EINVAL, "E=%d out of range [0, %d]", E, MXFP8_MAX_EXPERTS);
    if (N < 1 || K < 1) return fail(MXFP8_EINVAL, "N=%d and K=%d must be >= 1", N, K);
    if (M < 32 || (M % 32) != 0) return fail(MXFP8_EINVAL, "M=%lld must be a positive multiple of 32", (long long)M);
    if (M > (int64_t(1) << 31) - 256) return fail(MXFP8_EINVAL, "M=%lld too large", (long long)M);
    if (E == 0) return MXFP8_OK;
    if (!A || !sA || !B || !sB || !offs || !out) return fail(MXFP8_EINVAL, "null pointer argument");
    if (!aligned16(A) || !aligned16(B) || !aligned16(out))
        return fail(MXFP8_EALIGN, "A, B and out must be 16-byte aligned");
    if ((K % 8) != 0) return fail(MXFP8_EALIGN, "K=%d must be a multiple of 8 (16-byte output rows)", K);
    return MXFP8_OK;
}

// Scale factors the caller already laid out as tcgen05 blocks on the global
// 128-token grid (mxfp8_wgrad_grouped_sf), with the tiling they were laid out for.
struct SfUser {
    const uint8_t *sfA, *sfB;
    int kn, tn;
};

int run(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, const int32_t* offs, int E, int N,
        int K, int64_t M, uint16_t* out, void* ws, size_t ws_bytes, bool use_cache, void* stream,
        const SfUser* sfu = nullptr) {
    cudaEvent_t evb = g_ev_before, eva = g_ev_after;
    g_ev_before = g_ev_after = nullptr;
    const int stall = g_stall_next;
    g_stall_next = 0;
    int rc = validate(A, sA, B, sB, offs, E, N, K, M, out);
    if (rc) return rc;
    if (E == 0) return MXFP8_OK;
    mxw::TileConfig tc;
    mxw::WsLayout lay;
    if (sfu) {
        if (sfu->kn != 0 && sfu->kn != 1) return fail(MXFP8_EINVAL, "kn=%d must be 0 or 1", sfu->kn);
        if (!mxw::choose_tiles(N, K, E, M, sfu->kn + 1, sfu->tn, &tc))
            return fail(MXFP8_EINVAL, "tile rows tn=%d: a multiple of 16 in [16, %d]", sfu->tn, mxw::MAX_TN);
        if (!aligned16(sfu->sfA) || !aligned16(sfu->sfB))
            return fail(MXFP8_EALIGN, "sfA and sfB must be 16-byte aligned");
        const int64_t steps = (M + mxw::BK - 1) / mxw::BK;
        const int64_t rows_m = static_cast<int64_t>(tc.tiles_m) * steps * 2;
        const int64_t rows_n = static_cast<int64_t>(tc.tiles_n) * steps * tc.nblk_n;
        if (rows_m > (int64_t(1) << 31) - 1 || rows_n > (int64_t(1) << 31) - 1 ||
            static_cast<int64_t>(E) * tc.tiles_m * tc.tiles_n > (int64_t(1) << 31) - 1)
            return fail(MXFP8_EINVAL, "unsupported sizes");
        lay.tc = tc;
        lay.ts_max = static_cast<int>(steps);
        lay.plan_off = lay.sfm_off = lay.sfn_off = 0;
        lay.total = sizeof(int32_t) * (mxw::PLAN_HDR + 5 * static_cast<size_t>(E));
    } else if (!mxw::choose_tiles(N, K, E, M, orientation_mode(), tile_rows_setting(), &tc) ||
               !mxw::ws_layout(E, N, K, M, tc, &lay)) {
        return fail(MXFP8_EINVAL, "unsupported sizes");
    }
    if (!use_cache) {
        if (!ws) return fail(MXFP8_EINVAL, "null workspace");
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(MXFP8_EALIGN, "workspace must be 256-byte aligned");
        // the documented requirement (the bound over both orientations), not just
        // this call's layout, so that a size that works once works for any routing
        const size_t need = mxw::ws_bytes_any_orientation(E, N, K, M, tile_rows_setting());
        if (ws_bytes < need || ws_bytes < lay.total)
            return fail(MXFP8_ENOWS, "workspace of %zu bytes, need %zu", ws_bytes, need > lay.total ? need : lay.total);
    }
    int dev;
    DeviceInfo info;
    rc = current_device(&dev, &info);
    if (rc) return rc;
    {
        // Waiting warps park in mbarrier.try_wait (default hint 50 us; the
        // hardware resumes them when the phase completes) instead of spinning:
        // fewer issued instructions, less power, higher clocks under the power
        // cap. MXFP8_SUSPEND_NS overrides the hint (0 = plain polling). Set
        // once per device.
        static std::atomic<bool> hint_set[64];
        if (!hint_set[dev].load(std::memory_order_relaxed)) {
            const char* env = getenv("MXFP8_SUSPEND_NS");
            const long long ns = env ? atoll(env) : 50000;
            cudaError_t e = mxw::set_suspend_hint(static_cast<uint32_t>(ns < 0 ? 0 : (ns > 1000000 ? 1000000 : ns)));
            if (e != cudaSuccess) return fail_cuda(e, "suspend hint");
            hint_set[dev].store(true, std::memory_order_relaxed);
        }
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_cache) {
        rc = cached_workspace(dev, st, lay.total, &ws);
        if (rc) return rc;
    }
    // M side: 256-row pair tiles, 128 rows per CTA; N side: tn-row tiles, per CTA
    // n1/2 rows for the first MMA and n2/2 for the second
    CUtensorMap maps[6];
    const uint8_t* m_op = tc.kn ? B : A;
    const uint8_t* n_op = tc.kn ? A : B;
    const int n_rows = tc.kn ? N : K;
    rc = make_operand_map(&maps[0], m_op, tc.kn ? K : N, M, mxw::BM);
    if (rc) return rc;
    rc = make_operand_map3(&maps[1], n_op, M, n_rows, 1, tc.n1 / 2);
    if (rc) return rc;
    rc = make_operand_map3(&maps[2], n_op, M, n_rows, 1, tc.n2 ? tc.n2 / 2 : tc.n1 / 2);
    if (rc) return rc;
    // scale-factor blocks: the prep's re-layout in the workspace, or the caller's
    const uint8_t* sf_m = sfu ? (tc.kn ? sfu->sfB : sfu->sfA) : static_cast<uint8_t*>(ws) + lay.sfm_off;
    const uint8_t* sf_n = sfu ? (tc.kn ? sfu->sfA : sfu->sfB) : static_cast<uint8_t*>(ws) + lay.sfn_off;
    rc = make_sf_map(&maps[3], sf_m, static_cast<int64_t>(tc.tiles_m) * lay.ts_max * 2, 1);
    if (rc) return rc;
    rc = make_sf_map(&maps[4], sf_n, static_cast<int64_t>(tc.tiles_n) * lay.ts_max * tc.nblk_n, tc.nblk_n);
    if (rc) return rc;

    mxw::WgradArgs a;
    a.A = A; a.sA = sA; a.B = B; a.sB = sB; a.offs = offs;
    a.E = E; a.N = N; a.K = K; a.M = M; a.out = out;
    a.ws = static_cast<uint8_t*>(ws);
    a.lay = lay;
    a.dev = dev;
    a.num_sms = info.sms;
    a.wait_limit_ns = wait_limit_ns();
    a.stream = st;
    a.ev_before = evb;
    a.ev_after = eva;
    a.stall_first_stage = stall;
    a.grid = sfu ? 1 : MXW_GRID_KSTEPS;
    a.gather = sfu ? 0 : 1;
    // output as [E][N][K] for the TMA-store epilogue (used where its staging fits)
    a.tma_store = (store_mode() == 0 && make_out_map(&maps[5], out, K, N, E)) ? 1 : 0;
    if (!a.tma_store) maps[5] = maps[0];
    const char* what = "";
    cudaError_t e = mxw::launch_wgrad(a, maps, &what);
    if (e != cudaSuccess) return fail_cuda(e, what);
    return MXFP8_OK;
}

}  // namespace

int mxw::set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

extern "C" {

int mxfp8_wgrad_grouped(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                        const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out, void* stream) {
    return run(A, sA, B, sB, offs, E, N, K, M, out, nullptr, 0, true, stream);
}

size_t mxfp8_wgrad_workspace_bytes(int E, int N, int K, int64_t M) {
    return mxw::ws_bytes_any_orientation(E, N, K, M, tile_rows_setting());
}

int mxfp8_wgrad_set_tile_orientation(int mode) {
    if (mode < 0 || mode > 2) return fail(MXFP8_EINVAL, "tile orientation mode %d not in {0, 1, 2}", mode);
    g_orientation.store(mode, std::memory_order_relaxed);
    return MXFP8_OK;
}

int mxfp8_wgrad_set_epilogue_store(int mode) {
    if (mode < 0 || mode > 1) return fail(MXFP8_EINVAL, "epilogue store mode %d not in {0, 1}", mode);
    g_store_mode.store(mode, std::memory_order_relaxed);
    return MXFP8_OK;
}

int mxfp8_wgrad_set_tile_rows(int tn) {
    if (tn != 0 && (tn < 16 || tn > mxw::MAX_TN || tn % 16 != 0))
        return fail(MXFP8_EINVAL, "tile rows %d: 0 or a multiple of 16 in [16, %d]", tn, mxw::MAX_TN);
    g_tile_rows.store(tn, std::memory_order_relaxed);
    return MXFP8_OK;
}

int mxfp8_wgrad_tile_config(int E, int N, int K, int64_t M, int* kn, int* tn, int* tiles_m, int* tiles_n) {
    mxw::TileConfig tc;
    if (!kn || !tn || !tiles_m || !tiles_n) return fail(MXFP8_EINVAL, "null pointer argument");
    if (!mxw::choose_tiles(N, K, E, M, orientation_mode(), tile_rows_setting(), &tc))
        return fail(MXFP8_EINVAL, "N=%d and K=%d must be >= 1", N, K);
    *kn = tc.kn;
    *tn = tc.tn;
    *tiles_m = tc.tiles_m;
    *tiles_n = tc.tiles_n;
    return MXFP8_OK;
}

int mxfp8_wgrad_grouped_ws(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                           const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return run(A, sA, B, sB, offs, E, N, K, M, out, workspace, workspace_bytes, false, stream);
}

int mxfp8_wgrad_grouped_sf(const uint8_t* A, const uint8_t* sfA, const uint8_t* B, const uint8_t* sfB,
                           const int32_t* offs, int E, int N, int K, int64_t M, int kn, int tn, uint16_t* out,
                           void* stream) {
    const SfUser sfu{sfA, sfB, kn, tn};
    return run(A, sfA, B, sfB, offs, E, N, K, M, out, nullptr, 0, true, stream, &sfu);
}

size_t mxfp8_sf_blocks_bytes(int R, int64_t M, int tile_rows) {
    if (R < 1 || M < 32 || (M % 32) != 0 || tile_rows < 16 || (tile_rows % 16) != 0) return 0;
    const size_t tiles = (static_cast<size_t>(R) + tile_rows - 1) / tile_rows;
    const size_t steps = (static_cast<size_t>(M) + mxw::BK - 1) / mxw::BK;
    const size_t nblk = (static_cast<size_t>(tile_rows) + 127) / 128;
    return tiles * steps * nblk * mxw::SF_ATOM;
}

int mxfp8_quantize_tokenwise(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, void* stream) {
    if (R < 1) return fail(MXFP8_EINVAL, "R=%d must be >= 1", R);
    if (M < 32 || (M % 32) != 0) return fail(MXFP8_EINVAL, "M=%lld must be a positive multiple of 32", (long long)M);
    if (!x || !q || !s) return fail(MXFP8_EINVAL, "null pointer argument");
    if (!aligned16(x)) return fail(MXFP8_EALIGN, "x must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(q) & 7u) != 0) return fail(MXFP8_EALIGN, "q must be 8-byte aligned");
    int dev;
    DeviceInfo info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    cudaError_t e = mxw::launch_quantize(x, R, M, q, s, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "quantize kernel");
    return MXFP8_OK;
}

int mxfp8_grouped_gemm_tile_config(int E, int N, int K, int64_t M, int* tn, int* tiles_m_max, int* tiles_n) {
    if (!tn || !tiles_m_max || !tiles_n) return fail(MXFP8_EINVAL, "null pointer argument");
    mxw::TileConfig tc;
    mxw::GemmLayout lay;
    if (E < 1 || E > MXFP8_MAX_EXPERTS || N < 1 || (N % 8) != 0 || K < 32 || (K % 32) != 0 || M < 1 ||
        !mxw::choose_gemm_tiles(N, K, E, M, tile_rows_setting(), &tc) || !mxw::gemm_layout(E, N, K, M, tc, &lay))
        return fail(MXFP8_EINVAL, "unsupported sizes E=%d N=%d K=%d M=%lld", E, N, K, (long long)M);
    *tn = tc.tn;
    *tiles_m_max = lay.mtiles_max;
    *tiles_n = tc.tiles_n;
    return MXFP8_OK;
}

int mxfp8_grouped_gemm(const uint8_t* X, const uint8_t* sX, const uint8_t* W, const uint8_t* sW,
                       const int32_t* offs, int E, int64_t M, int N, int K, uint16_t* out, void* stream) {
    if (E < 1 || E > MXFP8_MAX_EXPERTS) return fail(MXFP8_EINVAL, "E=%d out of range [1, %d]", E, MXFP8_MAX_EXPERTS);
    if (M < 1 || M > (int64_t(1) << 31) - 1) return fail(MXFP8_EINVAL, "M=%lld out of range", (long long)M);
    if (N < 1) return fail(MXFP8_EINVAL, "N=%d must be >= 1", N);
    if (K < 32 || (K % 32) != 0) return fail(MXFP8_EINVAL, "K=%d must be a positive multiple of 32", K);
    if (!X || !sX || !W || !sW || !offs || !out) return fail(MXFP8_EINVAL, "null pointer argument");
    if (!aligned16(X) || !aligned16(W) || !aligned16(out))
        return fail(MXFP8_EALIGN, "X, W and out must be 16-byte aligned");
    if ((N % 8) != 0) return fail(MXFP8_EALIGN, "N=%d must be a multiple of 8 (16-byte output rows)", N);
    mxw::TileConfig tc;
    mxw::GemmLayout lay;
    if (!mxw::choose_gemm_tiles(N, K, E, M, tile_rows_setting(), &tc) || !mxw::gemm_layout(E, N, K, M, tc, &lay))
        return fail(MXFP8_EINVAL, "unsupported sizes");
    int dev;
    DeviceInfo info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    cudaEvent_t evb = g_ev_before, eva = g_ev_after;
    g_ev_before = g_ev_after = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    rc = cached_workspace(dev, st, lay.total, &ws);
    if (rc) return rc;
    // X: 256-row tiles, 128 rows per CTA; W as [E][N][K]: per CTA n1/2 rows for the
    // first MMA and n2/2 for the second
    CUtensorMap maps[6];
    rc = make_operand_map(&maps[0], X, static_cast<int>(M), K, mxw::BM);
    if (rc) return rc;
    rc = make_operand_map3(&maps[1], W, K, N, E, tc.n1 / 2);
    if (rc) return rc;
    rc = make_operand_map3(&maps[2], W, K, N, E, tc.n2 ? tc.n2 / 2 : tc.n1 / 2);
    if (rc) return rc;
    rc = make_sf_map(&maps[3], static_cast<uint8_t*>(ws) + lay.sfm_off,
                     static_cast<int64_t>(lay.mtiles_max) * lay.ksteps * 2, 1);
    if (rc) return rc;
    rc = make_sf_map(&maps[4], static_cast<uint8_t*>(ws) + lay.sfn_off,
                     static_cast<int64_t>(E) * tc.tiles_n * lay.ksteps * tc.nblk_n, tc.nblk_n);
    if (rc) return rc;
    mxw::GemmArgs a;
    a.X = X; a.sX = sX; a.W = W; a.sW = sW; a.offs = offs;
    a.E = E; a.N = N; a.K = K; a.M = M; a.out = out;
    a.ws = static_cast<uint8_t*>(ws);
    a.lay = lay;
    a.dev = dev;
    a.num_sms = info.sms;
    a.wait_limit_ns = wait_limit_ns();
    a.stream = st;
    a.ev_before = evb;
    a.ev_after = eva;
    // output as [1][M][N] for the TMA-store epilogue (used where its staging fits)
    a.tma_store = (store_mode() == 0 && make_out_map(&maps[5], out, N, M, 1)) ? 1 : 0;
    if (!a.tma_store) maps[5] = maps[0];
    const char* what = "";
    cudaError_t e = mxw::launch_gemm(a, maps, &what);
    if (e != cudaSuccess) return fail_cuda(e, what);
    return MXFP8_OK;
}

int mxfp8_quantize_transpose_bf16(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s, void* stream) {
    if (R < 1) return fail(MXFP8_EINVAL, "R=%d must be >= 1", R);
    if (M < 32 || (M % 32) != 0) return fail(MXFP8_EINVAL, "M=%lld must be a positive multiple of 32", (long long)M);
    if (!x || !q || !s) return fail(MXFP8_EINVAL, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(x) & 1u) != 0) return fail(MXFP8_EALIGN, "x must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return fail(MXFP8_EALIGN, "q must be 16-byte aligned");
    if (M / 64 + 1 > 0x7fffffffLL || (R + 127) / 128 > 65535)
        return fail(MXFP8_EINVAL, "M=%lld, R=%d: too large", (long long)M, R);
    int dev;
    DeviceInfo info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    cudaError_t e = mxw::launch_quantize_transpose(x, M, R, q, s, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "quantize-transpose kernel");
    return MXFP8_OK;
}

int mxfp8_quantize_transpose_bf16_sf(const uint16_t* x, int64_t M, int R, int tile_rows, uint8_t* q, uint8_t* s,
                                     uint8_t* sf, void* stream) {
    if (R < 1) return fail(MXFP8_EINVAL, "R=%d must be >= 1", R);
    if (M < 32 || (M % 32) != 0) return fail(MXFP8_EINVAL, "M=%lld must be a positive multiple of 32", (long long)M);
    if (tile_rows < 16 || (tile_rows % 16) != 0)
        return fail(MXFP8_EINVAL, "tile_rows=%d must be a positive multiple of 16", tile_rows);
    if (!x || !q || !sf) return fail(MXFP8_EINVAL, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(x) & 1u) != 0) return fail(MXFP8_EALIGN, "x must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return fail(MXFP8_EALIGN, "q must be 16-byte aligned");
    const int64_t rows = ((static_cast<int64_t>(R) + tile_rows - 1) / tile_rows) * tile_rows;
    if (M / 64 + 1 > 0x7fffffffLL || (rows + 127) / 128 > 65535 || rows > 0x7fffffffLL)
        return fail(MXFP8_EINVAL, "M=%lld, R=%d: too large", (long long)M, R);
    int dev;
    DeviceInfo info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    cudaError_t e = mxw::launch_quantize_transpose_sf(x, M, R, q, s, sf, tile_rows, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "quantize-transpose kernel");
    return MXFP8_OK;
}

const char* mxfp8_last_error(void) { return g_err; }

int mxfp8_device_status(int32_t* status, int clear) {
    if (!status) return fail(MXFP8_EINVAL, "null status pointer");
    cudaError_t e = mxw::read_device_status(status, clear);
    if (e != cudaSuccess) return fail_cuda(e, "device status");
    return MXFP8_OK;
}

// Failure-path test hook (not part of the public header): the next wgrad
// call on this thread declares 16 more bytes than its first pipeline stage
// receives, so that stage's wait can never complete and runs out after the
// configured limit (MXFP8_WAIT_LIMIT_MS). The kernel then stops its pipeline,
// sets MXFP8_DEV_WAIT_TIMEOUT and returns; nothing faults or hangs.
int mxfp8_test_stall_next_call(int enable) {
    g_stall_next = enable ? 1 : 0;
    return MXFP8_OK;
}

int mxfp8_wgrad_set_timing_events(void* ev_before, void* ev_after) {
    if ((ev_before == nullptr) != (ev_after == nullptr))
        return fail(MXFP8_EINVAL, "give both timing events or neither");
    g_ev_before = static_cast<cudaEvent_t>(ev_before);
    g_ev_after = static_cast<cudaEvent_t>(ev_after);
    return MXFP8_OK;
}

}  // extern "C"
