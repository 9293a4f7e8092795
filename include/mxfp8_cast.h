/*
 * mxfp8_cast.h -- C ABI of libmxfp8_cast.so: MX-FP8 (e4m3 elements, e8m0
 * block scales, blocks of 32) quantisation of bf16 matrices on sm_103a.
 *
 * Conventions for every entry point below
 *   - All data pointers are DEVICE pointers of the calling thread's current
 *     CUDA device (or managed memory), allocated and owned by the caller; the
 *     library allocates no device memory and keeps no pointer after the call
 *     returns.  Each pointer's memory type and device are checked on the
 *     host (MX_ERR_DEVICE), so a host pointer or another device's pointer is
 *     refused before any kernel sees it.  `stream` must belong to the same
 *     device.
 *   - Every pointer must be 16-byte aligned (int32 / int64 offset arrays:
 *     4- / 8-byte aligned), tensors are dense row-major with no padding.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; no call synchronises the device or reads
 *     device memory on the host.  Results are valid once the stream has
 *     executed the work.
 *   - Return value: MX_OK, or a negative MX_ERR_* code.  Argument errors are
 *     detected on the host before anything is enqueued (outputs untouched).
 *     MX_ERR_CUDA means a CUDA call failed; mx_last_cuda_error() has its code.
 *   - Calls that share an output buffer and run concurrently on the GPU race.
 *     Inputs and outputs of one call must not overlap.
 *   - Entry points may be called from several host threads at once: the only
 *     host state is a per-thread cache of TMA descriptors and per-device
 *     launch attributes set once.
 *
 * The rule, per 32-element block (OCP Microscaling Formats v1.0 conversion
 * with E4M3 elements and an E8M0 scale):
 *   amax  = max |x_i|
 *   scale byte s = clamp(floor(log2 amax) - 8, -127, 127) + 127; amax = 0
 *                  gives s = 0; a block holding Inf or NaN gives s = 0xFF
 *   q_i   = e4m3(x_i * 2^(127 - s)), round to nearest even, saturated to
 *           +-448 (e4m3 NaN for every element of an Inf/NaN block)
 * Directions (pytorch/ao PR #1869 "triton kernel to cast to mx across dim0
 * and dim1", summary):
 *   dim0: blocks along each row of X (M x K)    -> q0 (M x K) bytes
 *   dim1: blocks along each column of X         -> q1 (K x M) bytes, the
 *         row-major copy of X^T (X's column-major copy); q1[k][m] encodes
 *         X[m][k]
 * Blocked scale layout (the 128x4 layout of block-scaled GEMM scale factors;
 * 128x4 is the granularity named in pytorch/ao PR #3416 "[mxfp8 moe training]
 * parallelize along col blocks in scale blocked format kernel for groups
 * along K"): a scale matrix S (R x C) is padded with zeros to
 * ceil(R/128)*128 x ceil(C/4)*4, cut into 128x4 tiles stored one after
 * another in row-major tile order (512 bytes each), and S[r][c] sits at byte
 * (r%32)*16 + ((r%128)/32)*4 + c%4 of its tile.  Its size is
 * mx_blocked_bytes(R, C).
 */
#ifndef MXFP8_CAST_H
#define MXFP8_CAST_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MX_OK = 0,
  MX_ERR_NULL = -1,    /* a required pointer is NULL */
  MX_ERR_SHAPE = -2,   /* a size is zero, negative, too large or not a multiple of 32 */
  MX_ERR_ALIGN = -3,   /* a pointer is not suitably aligned */
  MX_ERR_CUDA = -4,    /* a CUDA call failed (see mx_last_cuda_error) */
  MX_ERR_GROUPS = -5,  /* invalid group count, or (device status) invalid offsets */
  MX_ERR_DEVICE = -6   /* a pointer is not device memory of the current device */
};

/* Fused dim0 + dim1 cast with both scale sets in blocked layout; one read of
 * X.  Defined by pytorch/ao PR #1869 "triton kernel to cast to mx across dim0
 * and dim1" (summary: read 32x32 tiles once, write the row-major and
 * column-major casts and their scales from each tile; future work: outer
 * tile 128, swizzled scales, coalesced writes).
 *   x       bf16 (M x K), row-major                      [in]
 *   M, K    M % 32 == 0, K % 32 == 0, 32 <= M, K <= 2^31 - 256
 *   q0      M x K bytes, e4m3, dim0                      [out]
 *   s0_blk  mx_blocked_bytes(M, K/32) bytes, e8m0        [out]
 *   q1      K x M bytes, e4m3, dim1                      [out]
 *   s1_blk  mx_blocked_bytes(K, M/32) bytes, e8m0        [out]
 * Padding bytes of the blocked buffers are written as zero. */
int mx_cast_dim0_dim1(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk, void* q1,
                      void* s1_blk, void* stream);

/* mx_cast_dim0_dim1 for callers that must not allocate device memory, with
 * its one piece of scratch in device memory reserved when the library is
 * loaded.  The pages have no counterpart: this is an entry point of this
 * library only.
 *
 * Who needs it: a process whose device memory is handed out by a caching
 * allocator that reserved it up front (a training or serving framework),
 * where an allocation from outside the pool can fail for lack of memory or
 * fragment it; and code that must not risk the device-wide synchronisation
 * an allocation can bring.  None of the entry points here allocate; this one
 * also keeps no per-stream state on the host: its scratch is one fixed
 * array instead of mx_cast_dim0_dim1's counter per stream.
 *
 * Arguments, layouts, output and errors as mx_cast_dim0_dim1, byte for byte.
 * The scratch is 256 bytes (64 words) of device memory, held by every GPU
 * that loads the library until the process exits; a call needs one word
 * (its tile-claim counter, for launches of 32 rounds of tiles or more), and
 * a call that would need more than 64 words is refused with MX_ERR_SHAPE.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Each call
 * clears the word it uses on the stream before its kernel.  All calls share
 * the array: calls whose kernels overlap on the GPU (different streams, no
 * ordering between them) race on it and give wrong output; order them on one
 * stream or with events. */
int mx_cast_dim0_dim1_noalloc(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk,
                              void* q1, void* s1_blk, void* stream);

/* dim1 cast only (the column-major copy and its blocked scales), as split out
 * of the fused kernel in the same pull request's follow-up (dim1 logic in its
 * own kernel).  Arguments as in mx_cast_dim0_dim1. */
int mx_cast_dim1(const void* x, int64_t M, int64_t K, void* q1, void* s1_blk, void* stream);

/* dim0 cast only (the row-major copy and its blocked scales): the dim0 half of
 * the fused kernel of pytorch/ao PR #1869 (summary), for callers that need
 * only the K-block copy (a forward-pass operand).
 *   x       bf16 (M x K), row-major                      [in]
 *   M, K    M >= 1 (any; dim0 blocks run along K), K % 32 == 0, K >= 32,
 *           M, K <= 2^31 - 256
 *   q0      M x K bytes, e4m3                            [out]
 *   s0_blk  mx_blocked_bytes(M, K/32) bytes, e8m0        [out]
 * Padding bytes of the blocked buffer are written as zero. */
int mx_cast_dim0(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk, void* stream);

/* Standalone conversion of a plain scale matrix to the blocked layout, the
 * operation of the scale-blocking kernels in pytorch/ao PR #3416 (Changes
 * list) and PR #2990 (perf analysis, scale swizzle kernels).
 *   s    R x C bytes, row-major, any alignment           [in]
 *   R, C >= 1, R <= 65535 * 128
 *   out  mx_blocked_bytes(R, C) bytes, 16-byte aligned   [out] */
int mx_scales_to_blocked(const void* s, int64_t R, int64_t C, void* out, void* stream);

/* Fused dim0 + dim1 cast of MoE activations with groups along M (pytorch/ao
 * PR #2990 "[mxfp8 moe training] add compile support": groups of rows given
 * by offsets; scale buffers sized by the bound rows + groups * 128 so that no
 * device-to-host read is needed).
 *   x            bf16 (M x K)                                   [in]
 *   M, K         M >= 1, K % 32 == 0, M, K <= 2^31 - 256
 *   offs         G int32 cumulative group ends (group g = rows
 *                [offs[g-1], offs[g]), offs[-1] = 0; offs[G-1] == M;
 *                empty groups allowed), device memory           [in]
 *   G            >= 1 (else MX_ERR_GROUPS)
 *   q0           M x K bytes: the ungrouped dim0 cast           [out]
 *   s0_blk       mx_grouped_m_scale_bytes(M, K, G, 0) bytes: group g's scale
 *                rows in blocked layout on their own, starting at row
 *                s0_row_offs[g] (byte s0_row_offs[g] * ceil4(K/32)) [out]
 *   s0_row_offs  G + 1 int64: sum over h < g of ceil(m_h/128)*128 [out]
 *   q1           K x M bytes: group g is the dim1 cast of its own rows
 *                (blocks of 32 start at the group's first row; the last
 *                block may be partial and counts missing rows as zero),
 *                in columns [offs[g-1], offs[g])                [out]
 *   s1_blk       mx_grouped_m_scale_bytes(M, K, G, 1) bytes: group g's
 *                (K x ceil(m_g/32)) scales in blocked layout on their own at
 *                byte ceil128(K) * s1_col_offs[g]                [out]
 *   s1_col_offs  G + 1 int64: sum over h < g of ceil(m_h/128)*4 [out]
 *   status       one int32, device memory: 0, or MX_ERR_GROUPS if the offsets
 *                are invalid (then nothing else is written)     [out]
 * Every byte of both scale buffers is written (padding zero). */
int mx_cast_grouped_m(const void* x, int64_t M, int64_t K, const int32_t* offs, int32_t G,
                      void* q0, void* s0_blk, int64_t* s0_row_offs, void* q1, void* s1_blk,
                      int64_t* s1_col_offs, int32_t* status, void* stream);

/* dim1 cast of 3D expert weights (pytorch/ao PR #2990, perf analysis: cast
 * the (E, N, K) weights as the reshaped 2D matrix (E*N, K) with the dim1
 * kernel, scales per expert).
 *   w       bf16 (E, N, K)                                       [in]
 *   E >= 1, N % 32 == 0, K % 32 == 0, E*N and K <= 2^31 - 256
 *   q1      K x (E*N) bytes: the dim1 cast of the (E*N, K) matrix;
 *           expert e owns columns [e*N, (e+1)*N)                  [out]
 *   s1_blk  mx_3d_scale_bytes(E, N, K) bytes: expert e's (K x N/32)
 *           scales in blocked layout at byte e * mx_blocked_bytes(K, N/32)
 *                                                                 [out] */
int mx_cast_3d_dim1(const void* w, int64_t E, int64_t N, int64_t K, void* q1, void* s1_blk,
                    void* stream);

/* dim0 cast of 3D expert weights: blocks of 32 along K, the direction the
 * forward pass reads the weights in.  The pages cast 3D weights only along N
 * with the dim1 kernel through the reshape to (E*N, K) (pytorch/ao PR #2990,
 * perf analysis); this applies the same reshape to the dim0 cast of PR #1869
 * and blocks each expert's scales on their own, like the dim1 variant.
 *   w       bf16 (E, N, K)                                       [in]
 *   E >= 1, N >= 1 (any), K % 32 == 0, K >= 32, E*N and K <= 2^31 - 256
 *   q0      E x N x K bytes: the dim0 cast of the (E*N, K) matrix [out]
 *   s0_blk  mx_3d_dim0_scale_bytes(E, N, K) bytes: expert e's (N x K/32)
 *           scales in blocked layout at byte e * mx_blocked_bytes(N, K/32);
 *           padding zero                                          [out] */
int mx_cast_3d_dim0(const void* w, int64_t E, int64_t N, int64_t K, void* q0, void* s0_blk,
                    void* stream);

/* Both directions of 3D expert weights in one read: mx_cast_3d_dim0's q0 and
 * s0_blk and mx_cast_3d_dim1's q1 and s1_blk (N % 32 == 0 required, as for
 * mx_cast_3d_dim1).  Buffer sizes as in those two calls. */
int mx_cast_3d_dim0_dim1(const void* w, int64_t E, int64_t N, int64_t K, void* q0, void* s0_blk,
                         void* q1, void* s1_blk, void* stream);

/* MX dequantisation to bf16.  The pages define no dequantisation kernel; the
 * value of an MX element is its scale times its element value (OCP
 * Microscaling Formats v1.0, MX block definition), here rounded once to bf16
 * (nearest even; subnormals kept; magnitudes rounding to 2^128 or more give
 * infinity; a NaN scale (0xFF) or NaN element gives NaN).  Applied to
 * (q0, s0_blk) of a cast it gives X back up to the cast's rounding; applied
 * to (q1, s1_blk), with R = K and C = M, it gives X^T.
 *   q       R x C bytes, e4m3, blocks of 32 along rows      [in]
 *   R, C    R >= 1, C % 32 == 0, C >= 32, R, C <= 2^31 - 256
 *   s_blk   mx_blocked_bytes(R, C/32) bytes, e8m0           [in]
 *   out     R x C bf16                                      [out] */
int mx_dequant_blocked(const void* q, int64_t R, int64_t C, const void* s_blk, void* out,
                       void* stream);

/* Tensorwise fp8: one dynamic scale for the whole tensor, the conversion of
 * pytorch/ao PR #1445 "[float8nocompile] Triton kernels for conversion to
 * float8 dtypes" (local amaxes in parallel, a global amax, then the
 * conversion, each block of which computes the scale itself).  Not an MX
 * format: the contrast case with a non-power-of-two scale.
 *   amax  = max |x|, written to *amax (fp32; NaN if x holds a NaN)
 *   scale = fp32 nearest to 448 / amax, written to *scale; amax = 0 gives
 *           1, a quotient beyond the largest finite fp32 gives that value
 *   q     = e4m3(fp32(x * scale)), nearest even, saturated to +-448
 *   x      n bf16 values, any shape, dense                    [in]
 *   n      >= 1, <= 2^40
 *   q      n bytes, e4m3                                      [out]
 *   scale  one fp32, device memory                            [out]
 *   amax   one fp32, device memory; also the call's reduction
 *          target (cleared, then reduced into)                [out]
 * Enqueues a 4-byte memset and two kernels. */
int mx_cast_tensorwise(const void* x, int64_t n, void* q, float* scale, float* amax,
                       void* stream);

/* Rowwise fp8: one scale per row, quantize_fp8_rowwise of the "FP8 linear
 * triton with row-wise scaling" gist.
 *   scale_r = bf16 nearest to max_j |x_rj| / 448 (bf16, the input's dtype)
 *   q_rj    = e4m3(fp32(x_rj / scale_r)), nearest even, saturated to +-448;
 *             a row whose scale is 0 (all zero, or amax below about 2^-125)
 *             gives signed zeros rather than the formula's 0/0
 *   x       bf16 (M x K)                                      [in]
 *   M, K    M >= 1, K >= 8, K % 8 == 0, M, K <= 2^31 - 256
 *   q       M x K bytes, e4m3                                 [out]
 *   scale   M bf16 values                                     [out] */
int mx_cast_rowwise(const void* x, int64_t M, int64_t K, void* q, void* scale, void* stream);

/* Size helpers (host only, no CUDA calls).  Return -1 for invalid sizes. */
int64_t mx_blocked_bytes(int64_t R, int64_t C);
/* dim 0: (M + 128*G) * ceil4(K/32); dim 1: ceil128(K) * (ceil(M/32) + 4*G). */
int64_t mx_grouped_m_scale_bytes(int64_t M, int64_t K, int32_t G, int32_t dim);
/* E * mx_blocked_bytes(K, N/32): dim1 scales of 3D weights. */
int64_t mx_3d_scale_bytes(int64_t E, int64_t N, int64_t K);
/* E * mx_blocked_bytes(N, K/32): dim0 scales of 3D weights. */
int64_t mx_3d_dim0_scale_bytes(int64_t E, int64_t N, int64_t K);

/* Text for an MX_* code (static storage). */
const char* mx_strerror(int code);

/* cudaError_t value of the last failed CUDA call made by this thread. */
int mx_last_cuda_error(void);

/* Device watchdog: every wait inside the kernels is bounded.  A CTA that
 * gives up stops all its roles, lets the copies it has in flight land, and
 * sets a device word (one per kernel file).  Returns the words OR-ed (0 or 1)
 * after synchronising the current device, clearing them if `clear` is
 * non-zero, or MX_ERR_CUDA. */
int mx_watchdog(int clear);

/* Bounds-checked builds (compiled with -DMX_DEBUG_BOUNDS): the number of
 * global stores the kernels refused because they would have left their
 * output buffer (each is skipped and counted, never trapped), cleared if
 * `clear` is non-zero.  The stand-in for a device memory checker.  Returns -1
 * in a release build (no checks compiled in), MX_ERR_CUDA if the count could
 * not be read.  Synchronises the current device. */
int mx_bounds_check(int clear);

/* Diagnostic for bounds-checked builds: one thread tries a 4-byte store just
 * past an 8-byte span over `buf16` (16 bytes of device memory owned by the
 * caller, 16-byte aligned); the check refuses it, leaves bytes 8..11
 * untouched and adds one to the count read by mx_bounds_check().  Returns
 * MX_OK, MX_ERR_NULL / MX_ERR_ALIGN / MX_ERR_DEVICE / MX_ERR_CUDA, or -1 in
 * a release build (nothing is launched). */
int mx_selftest_bounds(void* buf16, void* stream);

/* Diagnostic: enqueue one warp that waits, with a limit of `wait_ns`
 * nanoseconds (1e3 .. 1e10), on a barrier that nothing completes.  The wait
 * gives up, sets the watchdog word read by mx_watchdog() and the kernel
 * returns normally: the failure path of the bounded waits, exercised without
 * any fault.  Returns MX_OK, MX_ERR_SHAPE or MX_ERR_CUDA. */
int mx_selftest_watchdog(int64_t wait_ns, void* stream);

/* Diagnostic of checked builds (compiled with -DMX_DEBUG_BOUNDS, as
 * libmxfp8_cast_bounds.so): arm a stall for the calling thread's next launch
 * of a kernel whose waits are bounded (the cast kernels of mx_cast_dim0_dim1,
 * mx_cast_dim0, mx_cast_dim1, mx_cast_grouped_m and the 3D casts; the
 * bulk-staged kernel of mx_cast_rowwise, used for K <= 24576; the tiled
 * kernel of mx_dequant_blocked, used for C >= 1024).  In that launch the
 * thread of CTA 0 that issues its loads waits, at its `at`-th tile (rowwise:
 * step), on a barrier that nothing completes, for at most `wait_ns` nanoseconds
 * (1e3 .. 1e10).  The wait gives up, the CTA stops every role, lets the
 * copies it has in flight land, sets the word read by mx_watchdog(), and the
 * kernel returns normally: the abort path of a real cast, exercised without
 * any fault.  That launch's outputs are incomplete.  Without a kernel to take
 * it the stall stays armed; a launch consumes it.  Returns MX_OK,
 * MX_ERR_SHAPE (at < 0 or wait_ns out of range), or -1 in a release build,
 * whose kernels carry no stall hook (nothing is armed). */
int mx_selftest_arm_stall(int64_t at, int64_t wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_CAST_H */
