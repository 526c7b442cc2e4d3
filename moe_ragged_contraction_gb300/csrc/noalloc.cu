// Allocation-free variant of the weight-gradient entry point.
//
// Some callers may not allocate device memory themselves and have no
// workspace to hand over: for example a framework whose caching allocator owns
// the device heap and forbids allocations behind its back, or a process that
// reserved its device memory up front and must not call cudaMalloc afterwards.
// For them this file keeps the call's scratch (the schedule and the re-laid-out
// scale factors) in one fixed, file-scope device array that every GPU loading
// the library holds until the process exits.
#include <cstdio>
#include <mutex>

#include "mxw_internal.h"
#include "../../include/mxfp8_wgrad.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MXFP8_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current (in host code the array's name is only
// a host-side stand-in, never a device address).
int scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return MXFP8_ECUDA;
    if (dev < 0 || dev >= 64) return MXFP8_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return MXFP8_ECUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MXFP8_OK;
}

}  // namespace

extern "C" int mxfp8_wgrad_grouped_noalloc(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                                           const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out,
                                           void* stream) {
    if (E == 0) return mxfp8_wgrad_grouped_ws(A, sA, B, sB, offs, E, N, K, M, out, nullptr, 0, stream);
    const size_t need = mxfp8_wgrad_workspace_bytes(E, N, K, M);
    if (need > MXFP8_NOALLOC_SCRATCH_BYTES) {
        // (invalid sizes give need == 0 and are reported by the call below)
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "E=%d N=%d K=%d M=%lld need %zu bytes of scratch; the allocation-free entry point holds at most %zu",
                 E, N, K, (long long)M, need, (size_t)MXFP8_NOALLOC_SCRATCH_BYTES);
        return mxw::set_last_error(MXFP8_ENOWS, msg);
    }
    void* scratch = nullptr;
    int rc = scratch_on_current_device(&scratch);
    if (rc != MXFP8_OK) return mxw::set_last_error(rc, "cudaGetSymbolAddress failed for the scratch array");
    return mxfp8_wgrad_grouped_ws(A, sA, B, sB, offs, E, N, K, M, out, scratch, MXFP8_NOALLOC_SCRATCH_BYTES, stream);
}
