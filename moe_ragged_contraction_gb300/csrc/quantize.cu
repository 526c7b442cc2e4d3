// Tokenwise MXFP8 quantiser (input building only; not on the timed path).
//
// "Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on MI355X", section 1:
// the weight gradient's operands are quantised along the token axis, one E8M0
// scale per 32 tokens. Scale rule 2^ceil(log2(amax/448)), read exactly as the
// smallest integer e with amax <= 448 * 2^e (clamped to [-127, 127]; amax = 0
// gives -127), found from the bits of amax with no logarithm or division.
#include <cuda_fp8.h>

#include "mxw_internal.h"

namespace mxw {

constexpr int QT_THREADS = 256;
constexpr int QT_TOKENS_PER_THREAD = 8;
constexpr int QT_TOKENS_PER_BLOCK = QT_THREADS * QT_TOKENS_PER_THREAD;

// Four consecutive threads cover one 32-token block: each loads 8 floats,
// the group shares amax through two shuffles, each writes its 8 E4M3 bytes,
// and the first of the four writes the scale byte.
__device__ __forceinline__ void quantize_group(const float* __restrict__ x, long long M, uint8_t* __restrict__ q,
                                               uint8_t* __restrict__ s, long long row) {
    const long long t0 = static_cast<long long>(blockIdx.x) * QT_TOKENS_PER_BLOCK +
                         static_cast<long long>(threadIdx.x) * QT_TOKENS_PER_THREAD;
    const bool active = t0 < M;  // M % 32 == 0: a 32-token group is all in or all out
    float v[8];
    uint32_t amax_bits = 0;
    if (active) {
        const float4* src = reinterpret_cast<const float4*>(x + row * M + t0);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7fffffffu);
    }
    // |x| ordered as unsigned bit patterns; NaN and Inf sort above every finite value
    amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 1));
    amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 2));
    if (!active) return;

    uint8_t* qdst = q + row * M + t0;
    const bool leader = (threadIdx.x & 3) == 0;
    if (amax_bits >= 0x7f800000u) {  // NaN or Inf in the block
        *reinterpret_cast<uint2*>(qdst) = make_uint2(0x7f7f7f7fu, 0x7f7f7f7fu);
        if (leader) s[row * (M / 32) + (t0 >> 5)] = 0xFF;
        return;
    }
    int e;
    const int eb = static_cast<int>(amax_bits >> 23);
    if (eb == 0) {
        e = -127;  // zero or subnormal amax: below 448 * 2^-127
    } else {
        // amax = 1.m * 2^(eb-127) = f * 2^(eb-126) with f = 1.m / 2 in [0.5, 1);
        // 448 = 0.875 * 2^9, so e = (eb - 126) - 9, plus one when f > 0.875 (1.m > 1.75)
        e = eb - 135 + ((amax_bits & 0x7fffffu) > 0x600000u ? 1 : 0);
        e = max(-127, min(127, e));
    }
    // 2^-e as an fp32 (e in [-127, 120] here, so the exponent field is in range)
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        const __nv_fp8x2_storage_t p0 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[i] * inv, v[i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t p1 =
            __nv_cvt_float2_to_fp8x2(make_float2(v[i + 4] * inv, v[i + 5] * inv), __NV_SATFINITE, __NV_E4M3);
        lo |= static_cast<uint32_t>(p0) << (8 * i);
        hi |= static_cast<uint32_t>(p1) << (8 * i);
    }
    *reinterpret_cast<uint2*>(qdst) = make_uint2(lo, hi);
    if (leader) s[row * (M / 32) + (t0 >> 5)] = static_cast<uint8_t>(e + 127);
}

// grid: x covers the tokens of a row, y strides over rows
__global__ void __launch_bounds__(QT_THREADS) quantize_tokenwise_kernel(const float* __restrict__ x, int R,
                                                                        long long M, uint8_t* __restrict__ q,
                                                                        uint8_t* __restrict__ s) {
    for (long long row = blockIdx.y; row < R; row += gridDim.y) quantize_group(x, M, q, s, row);
}

cudaError_t launch_quantize(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((M + QT_TOKENS_PER_BLOCK - 1) / QT_TOKENS_PER_BLOCK),
              static_cast<unsigned>(R < 65535 ? R : 65535));
    quantize_tokenwise_kernel<<<grid, QT_THREADS, 0, stream>>>(x, R, M, q, s);
    return cudaGetLastError();
}

}  // namespace mxw
