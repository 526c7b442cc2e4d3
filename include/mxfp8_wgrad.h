/*
 * mxfp8_wgrad.h — C ABI of the GB300 (sm_103a) ragged MXFP8 weight-gradient
 * grouped GEMM.
 *
 * The operation ("Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on
 * MI355X", section 1; "Group-GEMM in XLA", Part 3, "Contracting"):
 *
 *   for every expert g:  dW[g] = dY[g]^T . X[g]
 *
 * where the per-expert token offsets cut the CONTRACTION (token) axis. The
 * operands arrive pre-quantised to MXFP8 along the token axis: A = dY^T [N,M]
 * and B = X^T [K,M] hold E4M3 bytes with the token axis contiguous, and each
 * run of 32 tokens of a row shares one E8M0 scale, stored in the row-major
 * planes sA [N, M/32] and sB [K, M/32]. The output is dense bf16 [E,N,K]:
 *
 *   out[g,n,k] = bf16_rne( sum_{t in [lo_g, hi_g)} a(n,t) b(k,t) )
 *   a(n,t) = e4m3(A[n,t]) * 2^(sA[n,t/32] - 127),  b likewise,
 *   lo_0 = 0, lo_g = offs[g-1], hi_g = offs[g],
 *
 * accumulated in fp32 on the tensor cores and narrowed to bf16 with
 * round-to-nearest-even (same page, section 5.5). Every output tile is owned
 * by exactly one CTA for its whole reduction (same page, section 4): no
 * atomics, no split-K, bit-reproducible output.
 *
 * Conventions for every entry point below:
 *  - Pointers to operands, scales, offsets, outputs and workspaces are DEVICE
 *    pointers owned by the caller; the library keeps none of them after the
 *    call returns. All work is enqueued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and the call returns without synchronising.
 *  - Layouts are dense row-major with no padding: A [N][M], B [K][M] (bytes),
 *    sA [N][M/32], sB [K][M/32] (bytes), offs [E] (int32), out [E][N][K]
 *    (bf16 bit patterns), x [R][M] (fp32).
 *  - The return value is a status code (MXFP8_OK or a negative MXFP8_E*);
 *    mxfp8_last_error() gives a message for the last failure on the calling
 *    thread. Argument errors are detected on the host before anything is
 *    enqueued. Errors the device detects (invalid offsets, a pipeline wait
 *    that ran out) set bits of a device status word read by
 *    mxfp8_device_status().
 *  - Requires an sm_103 (GB300) device: the library is built for sm_103a
 *    only, and every entry point that touches the device returns
 *    MXFP8_EUNSUPPORTED on any other.
 */
#ifndef MXFP8_WGRAD_H
#define MXFP8_WGRAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define MXFP8_OK 0
#define MXFP8_EINVAL (-1)       /* null pointer, negative or zero size, M % 32 != 0, E too large */
#define MXFP8_EALIGN (-2)       /* a pointer not 16-byte aligned, or K % 8 != 0 */
#define MXFP8_ECUDA (-3)        /* a CUDA runtime/driver error (message attached) */
#define MXFP8_EUNSUPPORTED (-4) /* the current device is not an sm_103 (GB300) GPU */
#define MXFP8_ENOWS (-5)        /* caller workspace smaller than mxfp8_wgrad_workspace_bytes() */

/* Bits of the device status word (mxfp8_device_status). */
#define MXFP8_DEV_OFFS_UNSORTED 1   /* offs decreased somewhere; clamped to a non-decreasing sequence */
#define MXFP8_DEV_OFFS_RANGE 2      /* an offset < 0 or > M; clamped into [0, M] */
#define MXFP8_DEV_OFFS_ALIGN 4      /* an offset not a multiple of 32; rounded down */
#define MXFP8_DEV_WAIT_TIMEOUT 8    /* a pipeline wait ran out; the CTA stopped and its tile is undefined */

/* Largest expert count supported by one call. */
#define MXFP8_MAX_EXPERTS 2048

/*
 * Ragged MXFP8 weight gradient ("Ragged MXFP8 Weight Gradients", section 1;
 * operand layout A = dY^T [N,M], B = X^T [K,M], scale planes [N,M/32] and
 * [K,M/32]; offs records where each expert's run of tokens ends).
 *
 *   A    [N][M]   E4M3 bytes, 16-byte aligned
 *   sA   [N][M/32] E8M0 bytes
 *   B    [K][M]   E4M3 bytes, 16-byte aligned
 *   sB   [K][M/32] E8M0 bytes
 *   offs [E]      int32 inclusive group ends. Preconditions (not checked on
 *                 the host, which would need a synchronisation): non-decreasing,
 *                 multiples of 32, offs[E-1] <= M. The device clamps violations
 *                 into that form, so no access ever leaves the operands, and
 *                 sets MXFP8_DEV_OFFS_* bits. Empty groups are allowed and give
 *                 exact +0.0 slabs. Tokens in [offs[E-1], M) are never read
 *                 into the contraction and may hold anything (NaN padding).
 *   E    number of experts, 0 <= E <= MXFP8_MAX_EXPERTS (E == 0: no-op)
 *   N, K output rows / columns, >= 1; K % 8 == 0
 *   M    token count (columns of A and B), M % 32 == 0, M >= 32
 *   out  [E][N][K] bf16, 16-byte aligned; every element is written
 *   stream cudaStream_t
 *
 * Scratch space (the scale re-layout and the schedule) comes from a cache the
 * library keeps per (device, stream), grown with stream-ordered allocation and
 * reused across calls; calls on one stream are ordered, so they never share
 * scratch concurrently. While `stream` is being captured into a CUDA graph the
 * cache does not grow: a call needing more scratch than the stream already
 * holds returns MXFP8_ENOWS (with a message) and records nothing, so make the
 * same call once on that stream before capturing, or use
 * mxfp8_wgrad_grouped_ws.
 */
int mxfp8_wgrad_grouped(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                        const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out,
                        void* stream);

/* Bytes of scratch that mxfp8_wgrad_grouped_ws needs for these sizes (an upper
 * bound over every routing of M tokens into E groups and over both tile
 * orientations, for the current tile-width setting). 0 if the sizes are
 * invalid. Host-only, no CUDA call. */
size_t mxfp8_wgrad_workspace_bytes(int E, int N, int K, int64_t M);

/* As mxfp8_wgrad_grouped, with caller-provided scratch: `workspace` is a
 * device pointer, 256-byte aligned, of at least
 * mxfp8_wgrad_workspace_bytes(E,N,K,M) bytes (else MXFP8_ENOWS). The
 * workspace must not be used by any other work until this call's kernels have
 * finished on `stream`.
 *
 * This call allocates nothing, so it may be recorded by CUDA stream capture
 * once the same sizes have been run eagerly in the context (which loads the
 * kernels and sets their attributes): the graph holds its two kernel launches,
 * and every replay reads the operands, scales and offs anew from the same
 * buffers (tests/test_gpu_graph.py). */
int mxfp8_wgrad_grouped_ws(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                           const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Tokenwise MXFP8 quantiser, used to build operands ("Ragged MXFP8 Weight
 * Gradients", section 1: one E8M0 scale per 32 elements along the token axis).
 * For each row r and each 32-token block b with amax = max |x| over the block:
 *   e = the smallest integer with amax <= 448 * 2^e (the scale 2^ceil(log2(amax/448))),
 *       clamped to [-127, 127]; amax == 0 gives e = -127;
 *   s[r][b] = e + 127 (E8M0);
 *   q[r][t] = E4M3(x[r][t] * 2^-e), round to nearest even, saturating at +-448.
 * A block holding a NaN or an infinity gets s = 0xFF and q = 0x7F (NaN).
 *   x [R][M] fp32 (16-byte aligned), q [R][M] bytes (8-byte aligned),
 *   s [R][M/32] bytes; R >= 1, M >= 32, M % 32 == 0.
 */
int mxfp8_quantize_tokenwise(const float* x, int R, int64_t M, uint8_t* q, uint8_t* s, void* stream);

/*
 * MXFP8 grouped GEMM with ragged rows: the forward and data-gradient products
 * of the same expert layer ("Group-GEMM in XLA", Part 1, the non-contracting
 * ragged dot; the weight gradient above is its contracting form). The rows of
 * X are cut into E contiguous groups by offs, and every row t of group g
 * multiplies the weights of expert g:
 *
 *   out[t][n] = bf16_rne( sum_k x(t,k) w(g,n,k) ),
 *   x(t,k) = e4m3(X[t][k]) * 2^(sX[t][k/32] - 127),  w likewise from W[g][n][k],
 *
 * accumulated in fp32 on the tensor cores, every output tile owned by one CTA
 * pair (bit-reproducible). Forward: X = activations [M][K], W = expert weights
 * [E][N][K] (output features x input features). Data gradient: X = dY [M][N'],
 * W = the weights transposed per expert [E][K'][N'], both quantised along the
 * contracted axis.
 *
 *   X    [M][K]      E4M3 bytes, 16-byte aligned
 *   sX   [M][K/32]   E8M0 bytes
 *   W    [E][N][K]   E4M3 bytes, 16-byte aligned
 *   sW   [E][N][K/32] E8M0 bytes
 *   offs [E]         int32 inclusive group ends over the rows of X; any row
 *                    boundaries (no 32-alignment needed: the scale blocks run
 *                    along k). Preconditions as for mxfp8_wgrad_grouped
 *                    (non-decreasing, <= M; clamped on the device and flagged
 *                    with MXFP8_DEV_OFFS_* otherwise). Rows at or past
 *                    offs[E-1] are written as +0.0.
 *   E    1..MXFP8_MAX_EXPERTS;  M rows (>= 1);  N >= 1, N % 8 == 0;  K >= 32, K % 32 == 0
 *   out  [M][N] bf16, 16-byte aligned; every element is written
 *
 * Scratch comes from the same per-(device, stream) cache as
 * mxfp8_wgrad_grouped, with the same rule under stream capture (no growth
 * while the stream is captured). The tile width follows mxfp8_wgrad_set_tile_rows
 * (the 256-row side is always on the rows of X).
 */
int mxfp8_grouped_gemm(const uint8_t* X, const uint8_t* sX, const uint8_t* W, const uint8_t* sW,
                       const int32_t* offs, int E, int64_t M, int N, int K, uint16_t* out, void* stream);

/*
 * Tiling mxfp8_grouped_gemm would use for these sizes under the current
 * settings: *tn = TN (output columns per tile), *tiles_m_max = the bound on
 * 256-row tiles over all routings (ceil(M/256) + E), *tiles_n = column tiles
 * per expert. Host-only, no CUDA call; MXFP8_EINVAL for sizes the entry point
 * rejects or null pointers.
 */
int mxfp8_grouped_gemm_tile_config(int E, int N, int K, int64_t M, int* tn, int* tiles_m_max, int* tiles_n);

/*
 * Fused quantise-and-transpose from token-major bf16 (the layout in which the
 * forward and backward passes produce dY and X): x [M][R] bf16 (bit patterns,
 * 2-byte aligned) becomes q [R][M] E4M3 with the token axis contiguous
 * (16-byte aligned) and s [R][M/32] E8M0, by the rule of
 * mxfp8_quantize_tokenwise applied to the transpose: the operand layout of
 * mxfp8_wgrad_grouped in one pass ("Ragged MXFP8 Weight Gradients", section 1:
 * operands quantised along the token axis; quantisation itself is outside the
 * timed operation there). R >= 1, M >= 32, M % 32 == 0.
 */
int mxfp8_quantize_transpose_bf16(const uint16_t* x, int64_t M, int R, uint8_t* q, uint8_t* s, void* stream);

/*
 * Scale factors written straight into the tensor core's layout ("Ragged MXFP8
 * Weight Gradients", section 5.6: the scale planes are pre-shuffled into the
 * form the matrix instruction reads; here the quantiser writes that form, so
 * the weight gradient below needs no re-layout pass).
 *
 * Layout ("SF blocks") for a [R][M] operand cut into tiles of `tile_rows` rows
 * and into 128-token steps on the global token grid: one 512-byte block per
 * (tile t, step g, 128-row block h of the tile), stored at
 *   ((t * ceil(M/128) + g) * ceil(tile_rows/128) + h) * 512,
 * holding tile row 128 h + r (r < 128) and 32-token block kb (kb < 4) of step
 * g at byte (r % 32) * 16 + (r / 32) * 4 + kb. Rows past R and tokens past M
 * hold 0x00.
 *
 * mxfp8_sf_blocks_bytes gives the size: ceil(R/tile_rows) * ceil(M/128) *
 * ceil(tile_rows/128) * 512 (0 for invalid sizes: R >= 1, M >= 32,
 * M % 32 == 0, tile_rows a positive multiple of 16). Host-only.
 */
size_t mxfp8_sf_blocks_bytes(int R, int64_t M, int tile_rows);

/*
 * mxfp8_quantize_transpose_bf16 that also writes the scales as SF blocks for
 * tiles of `tile_rows` rows (sf, mxfp8_sf_blocks_bytes(R, M, tile_rows) bytes,
 * every byte written); s may be NULL (no row-major plane). Arguments,
 * rounding and alignment otherwise as mxfp8_quantize_transpose_bf16.
 */
int mxfp8_quantize_transpose_bf16_sf(const uint16_t* x, int64_t M, int R, int tile_rows, uint8_t* q, uint8_t* s,
                                     uint8_t* sf, void* stream);

/*
 * The weight gradient of mxfp8_wgrad_grouped with the scales given as SF
 * blocks (no scale re-layout inside the call; the plan of the runs is still
 * built from offs on the device). The caller picks the tiling and lays the
 * scales out for it: kn = 0 puts the pair tile's 256-row side on A and tn
 * rows on B, kn = 1 the reverse (mxfp8_wgrad_tile_config reports the
 * library's choice); sfA holds A's scales as SF blocks for tiles of
 * (kn ? tn : 256) rows and sfB B's for tiles of (kn ? 256 : tn) rows, both
 * 16-byte aligned and at least mxfp8_sf_blocks_bytes(N, M, kn ? tn : 256)
 * and mxfp8_sf_blocks_bytes(K, M, kn ? 256 : tn) bytes long (the kernels
 * read that much; the host cannot check the allocations' sizes). tn is a multiple of 16 in [16, 448] (MXFP8_EINVAL
 * otherwise). Each expert's K-steps run on the 128-token grid: a run that
 * starts inside a step skips that step's leading 32-token chunks, so every
 * output element sums the same 32-token block products in the same order as
 * mxfp8_wgrad_grouped: the results are the same bits. Other arguments,
 * preconditions, scratch (the plan only) and errors as mxfp8_wgrad_grouped.
 */
int mxfp8_wgrad_grouped_sf(const uint8_t* A, const uint8_t* sfA, const uint8_t* B, const uint8_t* sfB,
                           const int32_t* offs, int E, int N, int K, int64_t M, int kn, int tn, uint16_t* out,
                           void* stream);

/* Message for the last non-zero status returned on the calling thread
 * (thread-local; never NULL). */
const char* mxfp8_last_error(void);

/* Reads the device status word of the current device into *status (a
 * combination of MXFP8_DEV_* bits; 0 when nothing was flagged) and, if
 * `clear` is non-zero, resets it. Synchronises the current device first. */
int mxfp8_device_status(int32_t* status, int clear);

/* Capacity of the allocation-free entry point's scratch array (32 MiB). */
#define MXFP8_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Allocation-free variant of mxfp8_wgrad_grouped. The paper has no
 * counterpart: this is an interface for callers that must not allocate. Some callers
 * cannot call cudaMalloc and have no workspace to pass: a framework whose own
 * caching allocator owns the device heap and forbids allocations behind its
 * back, or a process that reserves its device memory up front and may not
 * allocate afterwards. This entry point allocates nothing: it calls no
 * cudaMalloc, cudaFree or allocating library routine. Its scratch (schedule
 * and re-laid-out scale factors) lives in one fixed file-scope device array of
 * MXFP8_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library holds
 * until the process exits.
 *
 * Arguments, layouts, preconditions and results are those of
 * mxfp8_wgrad_grouped; the caller still provides A, sA, B, sB, offs and out.
 * Sizes whose scratch (mxfp8_wgrad_workspace_bytes) exceeds
 * MXFP8_NOALLOC_SCRATCH_BYTES are rejected with MXFP8_ENOWS and a message,
 * before any work is enqueued (e.g. the 16B shapes fit; the 671B shapes do not).
 *
 * Set-up: the CUDA runtime loads device code lazily, so the array (and the
 * kernels' code) is placed in device memory when first used in a CUDA
 * context. This entry point's first call in each context does that set-up: it
 * loads both and looks up the array's device address with that context
 * current (cudaGetSymbolAddress). That first call is the one moment it
 * commits device memory (the array's 32 MiB); every later call in the context
 * allocates nothing. A call with E == 0 (and valid N, K, M; the pointers are
 * not used) performs only the set-up: make it before reserving the rest of
 * the device's memory, and before any stream capture.
 *
 * Every call in a context shares the one array, and the array keeps whatever
 * the last call left in it (each call rewrites all the scratch it reads, so
 * nothing needs clearing): calls whose work overlaps on the GPU (different
 * streams, no ordering between them) race on it and must be avoided by the
 * caller.
 */
int mxfp8_wgrad_grouped_noalloc(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                                const int32_t* offs, int E, int N, int K, int64_t M, uint16_t* out,
                                void* stream);

/*
 * Output tiling. One CTA pair (two SMs) owns a 256 x TN tile of one expert's
 * output for the expert's whole token run. The 256-row side runs over the rows
 * of A (output rows n, TN over output columns k) or over the rows of B (output
 * columns k, TN over output rows n; the tile is then accumulated transposed
 * and stored back transposed). TN is a multiple of 16 up to 448. By default
 * the library picks the orientation and TN from a cost model of its kernel
 * (operand bytes per step against tensor-core cycles, padding and tile count).
 * The arithmetic per output element is the same for every tiling: results are
 * identical bit for bit across orientations and tile widths.
 *
 * mxfp8_wgrad_set_tile_orientation(mode) sets the orientation for the process
 * (every thread, every later call): 0 = automatic, 1 = 256 side on A,
 * 2 = 256 side on B. The initial mode comes from the environment variable
 * MXFP8_TILE_ORIENTATION ("auto", "nk" = 1, "kn" = 2), read at the first call.
 * mxfp8_wgrad_set_tile_rows(tn) forces TN (a multiple of 16 in [16, 448]) or
 * returns to the modelled choice (0). Both return MXFP8_EINVAL for other
 * values. mxfp8_wgrad_workspace_bytes follows the current settings: change
 * them before sizing a workspace.
 *
 * mxfp8_wgrad_tile_config(E, N, K, M, ...) reports the tiling the current
 * settings give for these sizes: *kn = 1 when the 256 side is on B, *tn = TN,
 * and the tile counts along the 256 side and the TN side. Host-only, no CUDA
 * call.
 */
int mxfp8_wgrad_set_tile_orientation(int mode);
int mxfp8_wgrad_set_tile_rows(int tn);
int mxfp8_wgrad_tile_config(int E, int N, int K, int64_t M, int* kn, int* tn, int* tiles_m, int* tiles_n);

/*
 * Epilogue stores (process-wide, every later call of mxfp8_wgrad_grouped{,_ws,
 * _noalloc} and mxfp8_grouped_gemm): mode 0 (default) narrows each 32 x 32
 * block of the accumulator into a shared-memory staging buffer and writes it
 * with a TMA store, wherever the staging fits beside the operand pipeline
 * without costing a stage (out 16-byte aligned, output rows a multiple of 8
 * elements; either orientation of the weight gradient's tiles, the 256-row
 * side on X in the grouped GEMM); blocks that straddle a tile, group or output
 * edge, and all other tilings, store straight from registers. Mode 1 stores
 * straight from registers always. The results are the same bits either way.
 * The initial mode comes from MXFP8_EPILOGUE_STORE ("auto" or "direct").
 * MXFP8_EINVAL for other modes.
 */
int mxfp8_wgrad_set_epilogue_store(int mode);

/* Measurement hook: when both events are non-NULL, the next
 * mxfp8_wgrad_grouped{,_ws} call on this thread records `ev_before` on its
 * stream right before the main contraction kernel and `ev_after` right after
 * it (cudaEvent_t handles). The hook is consumed by that one call. */
int mxfp8_wgrad_set_timing_events(void* ev_before, void* ev_after);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_WGRAD_H */
