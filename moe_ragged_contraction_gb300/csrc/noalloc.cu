// Allocation-free variant of the weight-gradient entry point.
//
// Some callers may not allocate device memory themselves and have no
// workspace to hand over: for example a framework whose caching allocator owns
// the device heap and forbids allocations behind its back, or a process that
// reserved its device memory up front and must not call cudaMalloc afterwards.
// For them this file keeps the call's scratch (the schedule and the re-laid-out
// scale factors) in one fixed, file-scope device array that every GPU loading
// the library holds until the process exits.
//
// The CUDA runtime loads device code lazily by default: the array is placed
// in device memory when this file's module is first used on a device, and the
// kernels' own module when one of them is first used. The set-up below does
// both, so that is the one moment this entry point commits device memory (the
// array's 32 MiB and the kernels' code). It runs on the first call in each
// CUDA context (a call with E = 0 does only the set-up), after which no call
// allocates anything.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "mxw_internal.h"
#include "../../include/mxfp8_wgrad.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MXFP8_NOALLOC_SCRATCH_BYTES];

// Device address of the array per CUDA context (an address from
// cudaGetSymbolAddress belongs to the context that was current when it was
// taken; in host code the array's name is only a host-side stand-in, never a
// device address).
struct CtxScratch {
    CUcontext ctx;
    void* ptr;
};
std::mutex g_noalloc_mu;
CtxScratch g_noalloc_cache[64] = {};
int g_noalloc_used = 0;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;

int setup_error(const char* what, cudaError_t e) {
    char msg[256];
    snprintf(msg, sizeof(msg), "allocation-free entry point set-up: %s failed: %s (%s)", what, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return mxw::set_last_error(MXFP8_ECUDA, msg);
}

// The scratch array's device address in the current context; the first call
// in a context also loads the kernels' module (see above).
int scratch_in_current_context(void** out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_ctx_current) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return setup_error("looking up cuCtxGetCurrent", e != cudaSuccess ? e : cudaErrorSymbolNotFound);
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return setup_error("cuCtxGetCurrent", cudaErrorDeviceUninitialized);
    void* p = nullptr;
    cudaError_t e = cudaSuccess;
    if (!ctx) {
        // no context current yet: the runtime binds the device's primary
        // context on its first call, this one
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return setup_error("cudaGetSymbolAddress of the scratch array", e);
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx)
            return setup_error("cuCtxGetCurrent", cudaErrorDeviceUninitialized);
    }
    for (int i = 0; i < g_noalloc_used; ++i)
        if (g_noalloc_cache[i].ctx == ctx) {
            *out = g_noalloc_cache[i].ptr;
            return MXFP8_OK;
        }
    if (g_noalloc_used == 64) return mxw::set_last_error(MXFP8_EUNSUPPORTED, "more than 64 CUDA contexts");
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return setup_error("cudaGetSymbolAddress of the scratch array", e);
    }
    e = mxw::load_kernel_modules();
    if (e != cudaSuccess) return setup_error("loading the kernels", e);
    g_noalloc_cache[g_noalloc_used++] = CtxScratch{ctx, p};
    *out = p;
    return MXFP8_OK;
}

}  // namespace

extern "C" int mxfp8_wgrad_grouped_noalloc(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                                           const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out,
                                           void* stream) {
    if (E != 0) {
        const size_t need = mxfp8_wgrad_workspace_bytes(E, N, K, M);
        if (need > MXFP8_NOALLOC_SCRATCH_BYTES) {
            // (invalid sizes give need == 0 and are reported by the call below)
            char msg[200];
            snprintf(msg, sizeof(msg),
                     "E=%d N=%d K=%d M=%lld need %zu bytes of scratch; the allocation-free entry point holds at most %zu",
                     E, N, K, (long long)M, need, (size_t)MXFP8_NOALLOC_SCRATCH_BYTES);
            return mxw::set_last_error(MXFP8_ENOWS, msg);
        }
    }
    void* scratch = nullptr;
    const int rc = scratch_in_current_context(&scratch);
    if (rc != MXFP8_OK) return rc;
    return mxfp8_wgrad_grouped_ws(A, sA, B, sB, offs, E, N, K, M, out, scratch, MXFP8_NOALLOC_SCRATCH_BYTES, stream);
}
