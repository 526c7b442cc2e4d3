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

// Scale exponent of a 32-element block from the bit pattern of its amax
// (finite): the smallest e with amax <= 448 * 2^e, clamped to [-127, 127].
__device__ __forceinline__ int block_exponent(uint32_t amax_bits) {
    const int eb = static_cast<int>(amax_bits >> 23);
    if (eb == 0) return -127;  // zero or subnormal amax: below 448 * 2^-127
    // amax = 1.m * 2^(eb-127) = f * 2^(eb-126) with f = 1.m / 2 in [0.5, 1);
    // 448 = 0.875 * 2^9, so e = (eb - 126) - 9, plus one when f > 0.875 (1.m > 1.75)
    const int e = eb - 135 + ((amax_bits & 0x7fffffu) > 0x600000u ? 1 : 0);
    return max(-127, min(127, e));
}

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
    const int e = block_exponent(amax_bits);
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

// ------------------------------------------------------------------ fused transpose

// Quantise-and-transpose from token-major bf16: x [M][R] (the layout dY and X
// have in the forward and backward passes) to q [R][M] E4M3 with the token
// axis contiguous and s [R][M/32], by the same rule as above (bf16 values are
// exact in fp32). A block handles a tile of 128 tokens x 128 features in two
// phases, each laid out so that a warp's memory instruction touches few
// cache lines (the L1 pipeline, not DRAM, limited the first version):
//  * load + transpose: thread (fg = lane % 16, tg = 2 warp + lane / 16) loads
//    the 8 x 8 sub-block of tokens 8 tg .. +7 and features 8 fg .. +7 (one
//    16-byte piece per token: a warp's load covers two whole 256-byte token
//    rows), transposes it in registers with byte permutes and writes eight
//    16-byte pieces (feature rows 8 fg + j, piece tg) into shared memory;
//  * quantise: in each of two passes, thread (feature 16 warp + 8 pass +
//    lane % 8, 32-token block lane / 8) reads its 32 values, finds the block's
//    exponent and writes 32 E4M3 bytes and the scale byte: a warp's store
//    covers 8 features x 128 contiguous bytes.
// Shared rows are 256 bytes, 16-byte piece p of row r stored at piece
// p ^ (r % 8) ^ (r / 8 % 8): the eight lanes of each 16-byte access phase then
// hit eight different bank groups in both phases.
constexpr int QX_TOK = 128;
constexpr int QX_FEAT = 128;
constexpr int QX_THREADS = 256;

__device__ __forceinline__ int qx_piece(int row, int p) { return p ^ (row & 7) ^ ((row >> 3) & 7); }

// Scale-factor block output of the quantiser (f2: the scales written straight
// into the layout the tensor core reads). Rows are cut into tiles of
// `tile_rows` rows, tokens into 128-token steps on the global grid; block h of
// tile t at step g holds tile rows 128 h .. 128 h + 127, and its 512 bytes
// hold row r, 32-token block kb at byte (r % 32) * 16 + (r / 32) * 4 + kb.
// Rows past R and tokens past M are zero.
struct SfOut {
    uint8_t* sf;       // nullptr: no block output
    int tile_rows;     // rows per tile
    int nblk;          // 128-row blocks per tile: ceil(tile_rows / 128)
    long long steps;   // 128-token grid steps: ceil(M / 128)
    int rows_out;      // rows covered by the blocks: tiles * tile_rows
    int tiles;         // ceil(R / tile_rows)
    int dead;          // rows of a tile's last block past the tile: nblk * 128 - tile_rows
};

__device__ __forceinline__ void sf_store(const SfOut& o, int f, long long step, int kb, uint8_t v) {
    const int t = f / o.tile_rows;
    const int rt = f - t * o.tile_rows;
    const int h = rt >> 7, r = rt & 127;
    const size_t atom = (static_cast<size_t>(t) * o.steps + step) * o.nblk + h;
    o.sf[atom * 512 + (r & 31) * 16 + (r >> 5) * 4 + kb] = v;
}

__global__ void __launch_bounds__(QX_THREADS) quantize_transpose_bf16_kernel(const uint16_t* __restrict__ x,
                                                                             long long M, int R, int vec,
                                                                             uint8_t* __restrict__ q,
                                                                             uint8_t* __restrict__ s,
                                                                             const SfOut sfo) {
    extern __shared__ __align__(16) uint4 sT[];  // [QX_FEAT][16] pieces of 8 bf16 (tokens)
    const long long t0 = static_cast<long long>(blockIdx.x) * QX_TOK;
    const int f0 = blockIdx.y * QX_FEAT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        const int fg = lane & 15, tg = 2 * warp + (lane >> 4);
        const int fb = f0 + 8 * fg;
        uint32_t r[8][4];  // r[i][w]: features (2w, 2w+1) of token i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long tok = t0 + 8 * tg + i;
            const uint16_t* src = x + tok * R + fb;
            if (tok < M && (vec & 1) && fb + 8 <= R) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
                r[i][0] = w.x; r[i][1] = w.y; r[i][2] = w.z; r[i][3] = w.w;
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t lo = (tok < M && fb + 2 * w < R) ? __ldg(src + 2 * w) : 0u;
                    const uint32_t hi = (tok < M && fb + 2 * w + 1 < R) ? __ldg(src + 2 * w + 1) : 0u;
                    r[i][w] = lo | (hi << 16);
                }
            }
        }
        // feature j, tokens (2w', 2w'+1): the j%2 halves of r[2w'][j/2] and r[2w'+1][j/2]
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
            uint4 c;
            c.x = __byte_perm(r[0][j >> 1], r[1][j >> 1], sel);
            c.y = __byte_perm(r[2][j >> 1], r[3][j >> 1], sel);
            c.z = __byte_perm(r[4][j >> 1], r[5][j >> 1], sel);
            c.w = __byte_perm(r[6][j >> 1], r[7][j >> 1], sel);
            const int row = 8 * fg + j;
            sT[row * 16 + qx_piece(row, tg)] = c;
        }
    }
    __syncthreads();
    const int b = lane >> 3;                    // 32-token block of the tile
    const long long tb = t0 + 32 * b;           // its first token
    const long long step = t0 / QX_TOK;         // this block's 128-token grid step
    if (sfo.sf && sfo.dead > 0 && blockIdx.y == 0) {
        // rows of each tile's last 128-row block that lie past the tile map to
        // no feature: zero their four scale bytes (one aligned word per row)
        const int live = sfo.tile_rows - 128 * (sfo.nblk - 1);
        for (int i = threadIdx.x; i < sfo.tiles * sfo.dead; i += QX_THREADS) {
            const int t = i / sfo.dead;
            const int r = live + (i - t * sfo.dead);
            const size_t atom = (static_cast<size_t>(t) * sfo.steps + step) * sfo.nblk + (sfo.nblk - 1);
            *reinterpret_cast<uint32_t*>(sfo.sf + atom * 512 + (r & 31) * 16 + (r >> 5) * 4) = 0u;
        }
    }
    if (tb >= M || f0 >= R) {
        // tokens past M (M % 32 == 0: a block is all in or all out) or rows
        // past R: only zero scale-factor bytes to write
        if (sfo.sf) {
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int f = f0 + 16 * warp + 8 * pass + (lane & 7);
                if (f < sfo.rows_out) sf_store(sfo, f, step, b, 0);
            }
        }
        return;
    }
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int fl = 16 * warp + 8 * pass + (lane & 7);
        const int f = f0 + fl;
        if (f >= R) {
            if (sfo.sf && f < sfo.rows_out) sf_store(sfo, f, step, b, 0);
            continue;
        }
        float v[32];
        uint32_t amax_bits = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = sT[fl * 16 + qx_piece(fl, 4 * b + i)];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[8 * i + 2 * k] = __uint_as_float(ws[k] << 16);
                v[8 * i + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
            }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7fffffffu);
        uint8_t* qdst = q + static_cast<long long>(f) * M + tb;
        uint8_t* sdst = s ? s + static_cast<long long>(f) * (M / 32) + (tb >> 5) : nullptr;
        uint32_t w[8];
        uint8_t sbyte;
        if (amax_bits >= 0x7f800000u) {  // NaN or Inf in the block
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0x7f7f7f7fu;
            sbyte = 0xFF;
        } else {
            const int e = block_exponent(amax_bits);
            const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(v[4 * i] * inv, v[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
                w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            sbyte = static_cast<uint8_t>(e + 127);
        }
        if (vec & 2) {  // q 32-byte aligned: one full sector per store
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(qdst), "r"(w[0]),
                         "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                         : "memory");
        } else {
            reinterpret_cast<uint4*>(qdst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(qdst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        if (s) *sdst = sbyte;
        if (sfo.sf) sf_store(sfo, f, step, b, sbyte);
    }
}

cudaError_t launch_quantize_transpose(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s,
                                      cudaStream_t stream) {
    return launch_quantize_transpose_sf(x, M, R, q, s, nullptr, 0, stream);
}

cudaError_t launch_quantize_transpose_sf(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s, uint8_t* sf,
                                         int tile_rows, cudaStream_t stream) {
    SfOut sfo;
    sfo.sf = sf;
    sfo.tile_rows = tile_rows > 0 ? tile_rows : 128;
    sfo.nblk = (sfo.tile_rows + 127) / 128;
    sfo.steps = (M + QX_TOK - 1) / QX_TOK;
    const long long tiles = (R + sfo.tile_rows - 1) / sfo.tile_rows;
    sfo.rows_out = static_cast<int>(tiles * sfo.tile_rows);
    sfo.tiles = static_cast<int>(tiles);
    sfo.dead = sfo.nblk * 128 - sfo.tile_rows;
    // bit 0: 16-byte loads of x rows; bit 1: 32-byte stores of q (M % 32 == 0 keeps every block aligned)
    const int vec = (((reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (R % 8) == 0) ? 1 : 0) |
                    ((reinterpret_cast<uintptr_t>(q) & 31u) == 0 ? 2 : 0);
    const long long gx = (M + QX_TOK - 1) / QX_TOK;
    // with block output, the blocks past R cover the last tile's padding rows
    const int rows = sf ? (sfo.rows_out > R ? sfo.rows_out : R) : R;
    const int gy = (rows + QX_FEAT - 1) / QX_FEAT;
    if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
    constexpr size_t smem = sizeof(uint16_t) * QX_FEAT * QX_TOK;  // 32 KB
    quantize_transpose_bf16_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), QX_THREADS, smem,
                                     stream>>>(x, M, R, vec, q, s, sfo);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((M + QT_TOKENS_PER_BLOCK - 1) / QT_TOKENS_PER_BLOCK),
              static_cast<unsigned>(R < 65535 ? R : 65535));
    quantize_tokenwise_kernel<<<grid, QT_THREADS, 0, stream>>>(x, R, M, q, s);
    return cudaGetLastError();
}

}  // namespace mxw
